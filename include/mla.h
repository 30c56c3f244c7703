/*
 * mla.h -- C ABI of a B300 (sm_103a) library for the decode step of
 * Multi-head Latent Attention (MLA) in its weight-absorbed form.
 *
 * The operation is the one of "DeepSeek-V3" (ekkoxiao.github.io), section
 * "Multi-Head Latent Attention": every cached token holds a latent
 * c^KV (d_c = 512) and a RoPE key k^R (d_h^R = 64) shared by all heads
 * (sub-section "KeyValue"); a head i scores position j as
 *     s = (q^C . W_i^UK c_j + q^R . k^R_j) / sqrt(d_h + d_h^R),   d_h = 128
 * (sub-section "注意力计算"), which the sub-section "潜在向量的作用" rewrites as
 *     q~ = (W_i^UK)^T q^C,   s = (q~ . c_j + q^R . k^R_j) / sqrt(192),
 *     o = W_i^UV (sum_j a_j c_j)        with a = softmax_j(s).
 * The dimensions are fixed by "DeepSeek-V3 技术报告精读" (oopvo.github.io),
 * section "维度分解详解": qk_nope 128, qk_rope 64, v 128, kv_lora_rank 512.
 *
 * One decode step is five calls on one stream:
 *   mla_absorb_q -> mla_rope_apply (queries) -> mla_decode
 *   -> mla_splitkv_combine -> mla_up_project,
 * or three: mla_absorb_rope_q (the first two in one launch) -> mla_decode
 *   -> mla_combine_up_project (the last two, without storing o_lat).
 * The cache's k^R is rotated once, when it is written (mla_rope_apply on the
 * cache), because the pages cache the rotated key.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers to row-major, contiguous data,
 *     16-byte aligned.  bf16 values are passed as their 16-bit patterns.
 *   - The caller owns all memory.  The library never allocates or frees
 *     device memory and never synchronises, except in mla_read_status.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and may be captured in a CUDA graph.
 *   - Arguments are validated on the host first; on an error nothing is
 *     launched and the status is returned at once.  Errors found on the
 *     device (a sequence length out of range, a wait that timed out) are
 *     recorded in the decode workspace and returned by mla_read_status.
 *   - Query positions are 0-based: keys sit at 0..L_b-1 and query s of S at
 *     L_b - S + s, which sees keys 0..L_b - S + s.
 *   - Kernels after the first of a step start before their predecessor has
 *     finished (programmatic dependent launch).  Each waits for it before
 *     reading that kernel's output, but weights (W_UV, W^O, W^DKV, W^KR) may
 *     stream in earlier: a weight must not be written by the kernel launched
 *     immediately before the call that reads it on the same stream.
 *   - The library keeps, per device, the device properties, its function
 *     attributes and the address of its scratch array, found on the first
 *     call on that device.  After cudaDeviceReset on a device, no call of
 *     this library may run on that device again in the same process.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16; /* raw bf16 bit pattern */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, misalignment, bad size or stride */
  MLA_ERR_UNSUPPORTED = 2, /* a shape the library does not implement */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  MLA_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
  MLA_ERR_BAD_SEQLEN = 5,  /* device: some seqlens[b] < S or > Lmax */
  MLA_ERR_TIMEOUT = 6      /* device: a bounded wait inside a kernel ran out */
} mla_status;

/* Fixed dimensions of the layout. */
enum { MLA_D_C = 512, MLA_D_R = 64, MLA_D_QK = 576, MLA_D_H = 128, MLA_D_V = 128 };

/* Human-readable name of a status code (static string, never NULL). */
const char *mla_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int mla_version(void);

/*
 * Absorb the key up-projection into the query ("潜在向量的作用":
 * q~_{b,s,h} = (W_h^UK)^T q^C_{b,s,h}).  fp32 accumulation on the tensor
 * cores, result rounded to bf16.
 *   q_nope [B,S,H,128]  bf16, the content query q^C
 *   W_UK   [H,128,512]  bf16, W_UK[h][d][k] = row block h of W^UK
 *   q_cat  [B,S,H,576]  bf16 output; columns 0..511 are written, 512..575
 *                       are left untouched (mla_rope_apply fills them)
 * Requires 1 <= H <= 128, B*S >= 1.
 */
mla_status mla_absorb_q(const mla_bf16 *q_nope, const mla_bf16 *W_UK, mla_bf16 *q_cat, int B,
                        int S, int H, void *stream);

/*
 * mla_absorb_q and the query RoPE in one launch: q_cat[..., 0:512] =
 * (W_h^UK)^T q^C as mla_absorb_q, and q_cat[..., 512:576] = RoPE(q_rope) at
 * position seqlens[b] - S + s as mla_rope_apply(MLA_POS_QUERY) ("Query": the
 * decoupled query key q^R is rotated at the query's position).
 *   q_rope  [B,S,H,64] bf16 (pre-RoPE),  seqlens [B] int32 device,
 *   base    RoPE base (10000); other arguments as mla_absorb_q.
 * Rows whose position seqlens[b] - S + s is negative keep their rope columns.
 */
mla_status mla_absorb_rope_q(const mla_bf16 *q_nope, const mla_bf16 *q_rope, const mla_bf16 *W_UK,
                             const int32_t *seqlens, mla_bf16 *q_cat, int B, int S, int H,
                             float base, void *stream);

/* How mla_rope_apply finds the position of row n. */
typedef enum {
  MLA_POS_EXPLICIT = 0, /* pos_src = int32 positions [N] */
  MLA_POS_QUERY = 1,    /* pos_src = seqlens [N / group]; row n = b*group + s sits at
                           seqlens[b] - group + s (group = S); rows with a negative
                           position are left untouched */
  MLA_POS_CACHE = 2     /* pos_src = seqlens [N / group]; row n = b*group + j sits at j
                           (group = Lmax); rows with j >= seqlens[b] are left untouched */
} mla_pos_mode;

/*
 * Rotary position embedding ("YaRN 扩展": the j-th 2-D pair at position m
 * turns by m * theta_j), on interleaved pairs (x_{2i}, x_{2i+1}) with
 * theta_i = base^(-2i/64):  (x, y) -> (x cos - y sin, x sin + y cos).
 * Angles are formed and reduced in fp64, rotated in fp32, stored as bf16.
 *   x_in  : element (n, i, d) at x_in [n*in_stride_n  + i*in_stride_h  + d], d < 64
 *   x_out : element (n, i, d) at x_out[n*out_stride_n + i*out_stride_h + d]
 *           (x_out may equal x_in for an in-place rotation; strides in elements,
 *            multiples of 8)
 *   N rows of nh heads each; pos_mode / pos_src / group as in mla_pos_mode.
 * Queries: x_in = q_rope [B,S,H,64] (strides H*64, 64), x_out = q_cat + 512
 * (strides H*576, 576), N = B*S, nh = H, MLA_POS_QUERY, group = S.
 * Cache fill: x_in = x_out = k_R [B,Lmax,64] (strides 64, 0), N = B*Lmax,
 * nh = 1, MLA_POS_CACHE, group = Lmax.
 */
mla_status mla_rope_apply(const mla_bf16 *x_in, int64_t in_stride_n, int64_t in_stride_h,
                          mla_bf16 *x_out, int64_t out_stride_n, int64_t out_stride_h,
                          int64_t N, int nh, int pos_mode, const int32_t *pos_src, int group,
                          float base, void *stream);

/*
 * RoPE with caller-given frequencies instead of base^(-2i/64): the same as
 * mla_rope_apply, with theta[32] a HOST array of the 32 pair frequencies
 * (finite, > 0), read during the call.  Used for YaRN (below).
 */
mla_status mla_rope_apply_freq(const mla_bf16 *x_in, int64_t in_stride_n, int64_t in_stride_h,
                               mla_bf16 *x_out, int64_t out_stride_n, int64_t out_stride_h,
                               int64_t N, int nh, int pos_mode, const int32_t *pos_src, int group,
                               const double *theta, void *stream);

/* mla_absorb_rope_q with caller-given frequencies theta[32] (host array). */
mla_status mla_absorb_rope_q_freq(const mla_bf16 *q_nope, const mla_bf16 *q_rope,
                                  const mla_bf16 *W_UK, const int32_t *seqlens, mla_bf16 *q_cat,
                                  int B, int S, int H, const double *theta, void *stream);

/*
 * YaRN frequencies ("YaRN 扩展": theta'_j = (1 - g_j) theta_j / s + g_j theta_j,
 * g_j = 1 for the high-frequency pairs, 0 for the low-frequency ones; the
 * technical report's long-context setting is s = 40, alpha = 1, beta = 32 over
 * an original context of 4096).  g_j is taken linear in the number of turns
 * r_j = orig_len * theta_j / (2 pi) a pair makes over the original context,
 * clamped to [0, 1] between alpha and beta turns; theta_j = base^(-2j/64).
 * Host-only arithmetic; writes theta[0..31].  Returns MLA_OK or
 * MLA_ERR_INVALID_ARG.  Use the result for the queries' and the cache's RoPE
 * alike, and pass mla_rope_yarn_softmax_scale(s) as mla_decode's softmax_scale.
 */
int mla_rope_yarn_frequencies(double base, double s, double alpha, double beta, double orig_len,
                              double *theta);

/*
 * Softmax scale of the YaRN setting ("Long Context Extension" of the
 * technical report: the scores are multiplied by 0.1 ln s + 1; "YaRN 扩展"
 * applies the factor to the scores before the softmax):
 *     *scale = (0.1 ln s + 1) / sqrt(d_h + d_h^R) = (0.1 ln s + 1) / sqrt(192).
 * Host-only arithmetic in double precision.  Returns MLA_OK, or
 * MLA_ERR_INVALID_ARG (and leaves *scale alone) if s < 1, s is not finite or
 * scale is NULL.  s = 1 gives the plain 1/sqrt(192).
 */
int mla_rope_yarn_softmax_scale(double s, double *scale);

/*
 * Bytes of device workspace mla_decode needs for this shape on the current
 * device (it depends on the device's SM count).  0 if the shape is
 * unsupported or no device is present.  The workspace carries the device
 * status word, the split plan and the partial results that
 * mla_splitkv_combine reads.
 */
size_t mla_decode_workspace_size(int B, int S, int H);

/*
 * Latent-space attention of every (b, s, h) query row over its visible
 * cache rows ("注意力计算" with the absorbed score of "潜在向量的作用"):
 *   s_j = (q_cat[..,0:512] . c_KV[b,j] + q_cat[..,512:576] . k_R[b,j]) * softmax_scale
 *   o_lat = sum_j softmax(s)_j c_KV[b,j]      (j = 0 .. L_b - S + s)
 * The cache rows of a sequence are split over all SMs (split-KV); each split
 * k leaves in the workspace, per query row, its reference exponent m_k, its
 * weight sum l_k and its normalised latent mix U_k (fp16; values beyond the
 * fp16 range saturate), to be merged by mla_splitkv_combine (call it next,
 * with the same workspace).  The kernel works out the split plan itself.
 *   q_cat   [B,S,H,576]  bf16, absorbed + rotated queries
 *   c_kv    [B,Lmax,512] bf16 latent cache
 *   k_r     [B,Lmax,64]  bf16 rotated RoPE keys
 *   seqlens [B] int32 (device), S <= seqlens[b] <= Lmax; rows >= seqlens[b]
 *           of the cache are never read into a result (they may hold anything)
 *   softmax_scale: 1/sqrt(192) for the pages' model
 *   workspace: >= mla_decode_workspace_size(B, S, H) bytes, 256-byte aligned
 * Requires S in {1, 2}, 1 <= H <= 128.
 */
mla_status mla_decode(const mla_bf16 *q_cat, const mla_bf16 *c_kv, const mla_bf16 *k_r,
                      const int32_t *seqlens, int B, int S, int H, int Lmax, float softmax_scale,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Merge the split-KV partials left by mla_decode in `workspace`:
 *   o_lat = sum_k w_k U_k / sum_k w_k,  w_k = l_k 2^(m_k - M),  M = max_k m_k
 * which restores the single normalisation over all visible positions.
 *   o_lat [B,S,H,512] bf16 output.  B, S, H must match the mla_decode call.
 */
mla_status mla_splitkv_combine(const void *workspace, size_t workspace_bytes, mla_bf16 *o_lat,
                               int B, int S, int H, void *stream);

/*
 * Up-projection of the latent result ("潜在向量的作用": o = W^UV o_lat),
 * fp32 accumulation on the tensor cores, rounded to bf16.
 *   o_lat [B,S,H,512] bf16,  W_UV [H,128,512] bf16 (W_UV[h][v][k]),
 *   out   [B,S,H,128] bf16 output (per-head output before W^O).
 * W_UV is read before the kernel waits for the one launched before it, so it
 * must not be written by that kernel.
 */
mla_status mla_up_project(const mla_bf16 *o_lat, const mla_bf16 *W_UV, mla_bf16 *out, int B,
                          int S, int H, void *stream);

/*
 * mla_splitkv_combine followed by mla_up_project in one launch: the merged
 * latent rows of each head go straight into the up-projection's operand in
 * shared memory and o_lat is never stored.
 *   o = W_UV[h] (sum_k w_k U_k / sum_k w_k),  w_k = l_k 2^(m_k - M)
 * ("注意力计算": one softmax over all visible positions; "潜在向量的作用":
 * o = W^UV o_lat).  `workspace` as left by mla_decode; W_UV [H,128,512]
 * bf16; out [B,S,H,128] bf16.  B, S, H must match the mla_decode call.
 * W_UV is read before the kernel waits for the one launched before it, so it
 * must not be written by that kernel.  MLA_ERR_UNSUPPORTED if a sequence can
 * be split into more than 96 segments on this device (more than 96
 * co-resident decode clusters).
 */
mla_status mla_combine_up_project(const void *workspace, size_t workspace_bytes, const mla_bf16 *W_UV,
                                  mla_bf16 *out, int B, int S, int H, void *stream);

/*
 * Bytes of device workspace mla_cache_append needs (fp32 partial products of
 * the down-projection and a status word); 0 if the shape is unsupported.
 */
size_t mla_cache_append_workspace_size(int B, int S, int d);

/*
 * The cache entries of the step's new tokens ("KeyValue"):
 *   c_t^KV = W^DKV h_t,   k_t^R = RoPE_t(W^KR h_t),
 * fp32 accumulation on the tensor cores, the RoPE angle reduced in fp64, both
 * rounded to bf16 and written at the tokens' positions
 * t = seqlens[b] - S + s (so seqlens already counts the new tokens, as
 * mla_decode expects):
 *   h      [B,S,d]   bf16 hidden states of the new tokens, d a multiple of 64
 *   W_DKV  [512,d]   bf16,   W_KR [64,d] bf16
 *   c_kv   [B,Lmax,512] bf16, k_r [B,Lmax,64] bf16: rows t are written, no
 *          other row is touched
 *   theta  host [32] RoPE frequencies (mla_rope_yarn_frequencies), or NULL
 *          for theta_j = 10000^(-2j/64)
 *   workspace >= mla_cache_append_workspace_size(B, S, d) bytes, 256-byte
 *          aligned, zero-filled before its first use; its first word is a
 *          status word (mla_read_status): a position outside [0, Lmax) sets
 *          MLA_ERR_BAD_SEQLEN and skips the token.  Words 1 and 2 hold a
 *          grid-wide barrier that each call leaves as it found it; after a
 *          call that reported MLA_ERR_TIMEOUT, zero-fill the workspace again.
 * One cooperative launch when all of its CTAs fit on the device at once
 * (the finalize follows a grid-wide barrier), else two launches.
 * The weights are read before the kernel waits for the one launched before
 * it on the stream, so they must not be written by that kernel.
 */
mla_status mla_cache_append(const mla_bf16 *h, const mla_bf16 *W_DKV, const mla_bf16 *W_KR,
                            const int32_t *seqlens, mla_bf16 *c_kv, mla_bf16 *k_r, int B, int S, int d,
                            int Lmax, const double *theta, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * The attention layer's output projection, one token at a time:
 *     u[n] = W x[n]          (u [BS][d], W [d][K], x [BS][K], all bf16 row-major)
 * with fp32 accumulation on the tensor cores, rounded to bf16.  "DeepSeek-V3"
 * (ekkoxiao.github.io), "注意力计算": u_t = W^O [o_{t,1}; ...; o_{t,H}], so
 *   x = out of mla_up_project viewed as [BS][H * 128] and W = W^O [d][H * 128];
 * and, with the value up-projection absorbed into W^O ("DeepSeek-V3
 * 技术报告精读" (oopvo.github.io), "MLA"),
 *   x = o_lat viewed as [BS][H * 512] and W = W^O blockdiag(W_h^UV)
 *   [d][H * 512], a weight the caller forms once (4x the bytes of W^O for
 *   d_c = 512, d_v = 128, so the unfolded pair streams less per step).
 * Requires K and d multiples of 128.  workspace: at least
 * mla_output_project_workspace_size(BS, K, d) bytes, 256-byte aligned (may be
 * NULL when that size is 0); it holds fp32 partial products over slices of K,
 * summed in a fixed order by a second launch.  x is read after the kernel
 * launched before this one finishes; W may stream in before, so it must not
 * be written by that kernel.  Device-side errors go to the library status
 * word (mla_read_status(NULL, stream)).
 */
size_t mla_output_project_workspace_size(int BS, int K, int d);
mla_status mla_output_project(const mla_bf16 *x, const mla_bf16 *W, mla_bf16 *u, int BS, int K, int d,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prefill, step 1: the keys and values of every cached token expanded per
 * head ("KeyValue": k^C_{t,i} = W_i^UK c_t, v^C_{t,i} = W_i^UV c_t), fp32
 * accumulation on the tensor cores, rounded to bf16:
 *   c_kv  [B,Lmax,512] bf16 (every row is expanded; rows past a sequence's
 *         length may hold anything, mla_prefill_attention never uses them)
 *   W_UK, W_UV [H,128,512] bf16
 *   k_c, v_c   [B,Lmax,H,128] bf16 outputs
 * Requires 1 <= H <= 128 and B * Lmax < 2^31 - 128.  One launch.
 * Device-side errors go to the library status word.
 */
mla_status mla_prefill_expand(const mla_bf16 *c_kv, const mla_bf16 *W_UK, const mla_bf16 *W_UV,
                              mla_bf16 *k_c, mla_bf16 *v_c, int B, int Lmax, int H, void *stream);

/*
 * Prefill, step 2: causal attention of S new query positions per sequence
 * over the expanded keys and values ("注意力计算"):
 *   o_{t,h} = sum_{j <= t} a_j v^C_{j,h},
 *   a = softmax_j((q^C_{t,h} . k^C_{j,h} + q^R_{t,h} . k^R_j) * softmax_scale)
 * for query s of sequence b at position t = seqlens[b] - S + s (the mla_decode
 * rule; S = seqlens[b] is a whole prompt, a smaller S a chunk after cached
 * context), with fp32 scores, P rounded to bf16, fp32 accumulation:
 *   q_nope  [B,S,H,128] bf16,
 *   q_rope  [B,S,H,64] bf16, ALREADY rotated at the query positions
 *           (mla_rope_apply with MLA_POS_QUERY and group = S),
 *   k_c, v_c [B,Lmax,H,128] bf16 from mla_prefill_expand,
 *   k_r     [B,Lmax,64] bf16, the cache's rotated keys,
 *   seqlens [B] int32 device, S <= seqlens[b] <= Lmax,
 *   softmax_scale  1/sqrt(192) (or the YaRN factor times it),
 *   out     [B,S,H,128] bf16 output (per-head output before W^O).
 * Requires 1 <= H <= 128 and 1 <= S <= Lmax.  A sequence whose length is out
 * of range sets MLA_ERR_BAD_SEQLEN in the library status word and its rows of
 * `out` are not written.  Cache rows at or past seqlens[b] are never used,
 * whatever they hold.
 */
mla_status mla_prefill_attention(const mla_bf16 *q_nope, const mla_bf16 *q_rope, const mla_bf16 *k_c,
                                 const mla_bf16 *k_r, const mla_bf16 *v_c, const int32_t *seqlens, int B,
                                 int S, int H, int Lmax, float softmax_scale, mla_bf16 *out, void *stream);

/*
 * Test hook for the kernels' bounded waits.  The next mla_decode call (only
 * that one) launches with its split-plan barrier left incomplete: every warp
 * that waits on it gives up after wait_limit_ns nanoseconds (instead of the
 * usual 1 s), records MLA_ERR_TIMEOUT in the decode workspace and winds down
 * before issuing any copy or MMA; the call writes no partial result.  Later
 * calls are normal.  Returns MLA_ERR_INVALID_ARG unless 0 < wait_limit_ns <= 1e9.
 * The paper has no counterpart: it exists so that a test can show that a
 * wait that runs out is reported and leaves the device usable.
 */
mla_status mla_debug_decode_stall(uint64_t wait_limit_ns);

/*
 * Synchronise `stream`, return the device-side status recorded in
 * `workspace` by earlier mla_decode calls (MLA_OK, MLA_ERR_BAD_SEQLEN or
 * MLA_ERR_TIMEOUT; MLA_ERR_CUDA if the stream reports an error) and clear it.
 */
mla_status mla_read_status(void *workspace, void *stream);

/*
 * Allocation-free latent decode: mla_decode followed by mla_splitkv_combine,
 * with the split-KV workspace taken from a fixed scratch array inside the
 * library instead of from the caller.  The paper has no counterpart; this
 * entry exists for callers that cannot allocate device memory on their
 * decode path -- a serving process that reserves all of HBM for its own pool
 * up front, or a real-time loop that must not call cudaMalloc because it can
 * synchronise the device and stall other streams.
 *   q_cat, c_kv, k_r, seqlens, B, S, H, Lmax, softmax_scale: as mla_decode
 *   o_lat [B,S,H,512] bf16 output, as mla_splitkv_combine
 * Scratch: one MLA_STATIC_SCRATCH_BYTES array per device, reserved when the
 * library's device code is loaded on that device and held until the process
 * exits.  A shape is accepted when mla_decode_workspace_size(B, S, H) is at
 * most MLA_STATIC_SCRATCH_BYTES (32 MiB: e.g. B = 32, S = 1, H = 128 on a
 * 148-SM B300); a larger one returns MLA_ERR_WORKSPACE and launches nothing.
 * Every call on a device shares that one array and leaves its contents
 * behind; each call writes every scratch byte it reads before reading it, so
 * nothing has to be cleared between calls.  Calls whose kernels overlap on
 * the GPU (different streams, no ordering between them) race on the array
 * and give wrong results: order them on one stream.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.
 * Device-side errors go to the library status word, read by
 * mla_read_status(NULL, stream).  The call allocates and frees nothing.
 */
enum { MLA_STATIC_SCRATCH_BYTES = 32 << 20 };
mla_status mla_decode_noalloc(const mla_bf16 *q_cat, const mla_bf16 *c_kv, const mla_bf16 *k_r,
                              const int32_t *seqlens, int B, int S, int H, int Lmax,
                              float softmax_scale, mla_bf16 *o_lat, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
