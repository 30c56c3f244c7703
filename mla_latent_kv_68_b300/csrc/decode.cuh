// decode.cuh -- latent-space MLA decode over the compressed cache, split-KV.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention":
//   score   s_j = (q~ . c_j + q^R . k^R_j) / sqrt(d_h + d_h^R)   ("注意力计算",
//           with the absorbed content term of "潜在向量的作用")
//   softmax over the visible positions, aggregation in latent space
//           o_lat = sum_j a_j c_j                                   ("潜在向量的作用")
// All query rows of one sequence (S*H of them, up to 128 per "row block")
// share every cache tile, so one tile feeds two dense contractions:
//   S[128 x 64]   = Q[128 x 576] . K_tile[64 x 576]^T      (K = [c ; k^R])
//   O[128 x 512] += P[128 x 64]  . C_tile[64 x 512]
//
// B300 mapping.  The fp32 accumulator O (128 x 512) fills one SM's entire
// tensor memory, and Q (128 x 576 bf16) plus a cache tile do not fit one SM's
// shared memory next to it.  So each unit of work runs on a CLUSTER OF TWO
// CTAs on two SMs:
//   rank 0 ("score CTA"): Q lives in its tensor memory (288 columns) and is
//       the A operand of the QK^T MMAs (A-from-TMEM form); two 64-column S
//       buffers; it streams full 576-wide cache rows through a 3-stage TMA
//       ring, runs the online softmax and sends P (bf16, already in the
//       128-byte-swizzled MMA layout) and the per-row rescale factor into
//       rank 1's shared memory with asynchronous remote stores (st.async)
//       whose bytes complete a transaction-counted barrier there.
//   rank 1 ("value CTA"): O lives in all 512 columns of its tensor memory; it
//       streams the 512-wide c rows of the same tiles (they are L2 hits right
//       after rank 0's reads) and issues O += P . C with C read as an
//       MN-major operand straight from the TMA tile.
// Neither CTA duplicates the other's tensor work, and HBM sees each cache
// byte once.
//
// Online softmax (log2 domain, s2 = s * scale * log2 e).  Each row keeps an
// INTEGER reference exponent m and l = sum 2^(s2 - m) of the bf16-rounded
// weights it sent.  m moves only when a tile's maximum exceeds m + 8; then
// m := ceil(max) and O, l are scaled by alpha = 2^(m_old - m_new), an exact
// power of two, so the rescale adds no rounding.  Weights stay <= 2^8.
//
// Split-KV: the grid is G groups x (row blocks) clusters; group g owns a
// contiguous run of cache tiles over all sequences (splitkv.cuh).  Each
// segment (a sequence's share of a group's run) leaves O unnormalised plus
// (m, l) per row; splitkv.cuh merges them.
//
// Every wait is bounded (sm100.cuh).  A wait that runs out aborts the CTA's
// remaining work; the cluster peer notices through its own waits.  Both CTAs
// meet in a final cluster barrier so neither exits while the other may still
// touch its shared memory.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kDecThreads = 224;  // 7 warps
constexpr int kTok = 64;          // cache rows per tile
constexpr int kStages = 3;
constexpr int kBlk = kTok * 128;  // one 64-column block of a tile, bytes
constexpr int kStage0 = 9 * kBlk; // score CTA: 8 c blocks + 1 k^R block
constexpr int kStage1 = 8 * kBlk; // value CTA: 8 c blocks
constexpr int kOffP = kStages * kStage1;            // value CTA: P[2] (128 x 64 bf16 each)
constexpr int kPBytes = 128 * kTok * 2;
constexpr int kOffAlpha = kOffP + 2 * kPBytes;      // value CTA: alpha[2][128] f32
constexpr int kOffBar = kOffAlpha + 2 * 128 * 4;
constexpr int kNumBars = 21;
constexpr uint32_t kPTx = kPBytes + 128 * 4;  // bytes of one P slot + its alpha column
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kDecSmem = kOffMisc + 16;
static_assert(kStages * kStage0 <= kOffBar, "score CTA stages overlap the barriers");
static_assert(kDecSmem <= 232448, "decode shared memory exceeds 227 KB");
constexpr uint32_t kQCol = 128;  // score CTA: Q at tensor-memory columns 128..415

// barrier indices
enum : int {
  B_FULL = 0, B_EMPTY = 3,           // TMA ring (both CTAs)
  B_SFULL = 6, B_SEMPTY = 8,         // score CTA: S buffers
  B_PEMPTY = 10,                     // score CTA: P slot in the value CTA free again
  B_QREADY = 12,                     // score CTA: Q of the segment is in tensor memory
  B_PFULL = 13,                      // value CTA: P + alpha of a tile have arrived
  B_PREADY = 15,                     // value CTA: O rescaled, P may be consumed
  B_PVDONE = 17,                     // value CTA: P . C of a tile completed
  B_OFREE = 19,                      // value CTA: epilogue has read O
  B_DRAIN = 20                       // both: final MMA drain
};

struct DecodeParams {
  const __nv_bfloat16* q_cat;  // [B,S,H,576]
  const int32_t* seqlens;      // [B]
  const int32_t* prefix;       // plan (splitkv.cuh)
  const int32_t* gfirst;
  const int32_t* segbase;
  const int32_t* gstart;       // [G] first sequence of each group's run
  float2* ml;                  // [slots * n_rb, 128]        (m, l) per row
  float* opart;                // [slots * n_rb, 512, 128]   column-major O per segment
  uint32_t* status;
  const uint32_t* plan_ok;
  int B, S, H, Lmax, n_rb, G;
  float scale_log2;            // softmax_scale * log2(e)
  uint64_t timeout_ns;
};

struct TileInfo {
  int b, t, L, i, k, slot;
  bool first, last;
};

// Visit, in order, every cache tile of group g (see splitkv.cuh for the plan).
template <class F>
__device__ __forceinline__ void for_each_tile(const DecodeParams& p, int g, F&& f) {
  const int64_t T = p.prefix[p.B];
  if (T <= 0) return;
  const int64_t beg = (int64_t)g * T / p.G, end = (int64_t)(g + 1) * T / p.G;
  if (beg >= end) return;
  int i = 0, k = 0;
  for (int b = p.gstart[g]; b < p.B; ++b) {
    const int64_t x0 = p.prefix[b], x1 = p.prefix[b + 1];
    if (x0 >= end) break;
    if (x1 <= beg) continue;
    const int tb = (int)(max(beg, x0) - x0), te = (int)(min(end, x1) - x0);
    const int slot = p.segbase[b] + (g - p.gfirst[b]);
    const int L = p.seqlens[b];
    for (int t = tb; t < te; ++t, ++i) {
      const TileInfo ti{b, t, L, i, k, slot, t == tb, t == te - 1};
      if (!f(ti)) return;
    }
    ++k;
  }
}

// All 32 lanes wait; the outcome is made warp-uniform so that warp-collective
// tensor-memory instructions after it never run with a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// Exact 2^d for an integer d <= 0 (0 below the normal range).
__device__ __forceinline__ float exp2_int(int d) {
  return d <= -127 ? 0.f : __int_as_float((127 + d) << 23);
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_kr,
                  const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int rb = cluster % p.n_rb, g = cluster / p.n_rb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    if (smem_u32(smem) & 1023u) {  // the swizzled tiles need 1 KB alignment
      *abort_flag = 1u;
      atomicOr(p.status, kDevErrInternal);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar[B_FULL + s], 1);
      mbar_init(&bar[B_EMPTY + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_SFULL + s], 1);
      mbar_init(&bar[B_SEMPTY + s], 128);
      mbar_init(&bar[B_PEMPTY + s], 1);
      mbar_init(&bar[B_PFULL + s], 1);
      mbar_init(&bar[B_PREADY + s], 128);
      mbar_init(&bar[B_PVDONE + s], 1);
    }
    mbar_init(&bar[B_QREADY], 128);
    mbar_init(&bar[B_OFREE], 128);
    mbar_init(&bar[B_DRAIN], 1);
    if (rank == 1) {  // first phase of each P slot expects one slot's bytes
      mbar_arrive_expect_tx(&bar[B_PFULL + 0], kPTx);
      mbar_arrive_expect_tx(&bar[B_PFULL + 1], kPTx);
    }
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_kr);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them remotely
  const uint32_t tmem = *tmem_slot;
  const bool run = (*p.plan_ok != 0u) && (*abort_flag == 0u);

  if (run && warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t sbytes = rank == 0 ? kStage0 : kStage1;
      int last_use[kStages] = {-1, -1, -1};
      for_each_tile(p, g, [&](const TileInfo& ti) {
        const int st = ti.i % kStages;
        const uint32_t ph = (uint32_t)(ti.i / kStages) & 1u;
        if (!mbar_wait(&bar[B_EMPTY + st], ph ^ 1u, wc)) return false;
        uint8_t* dst = smem + st * sbytes;
        mbar_arrive_expect_tx(&bar[B_FULL + st], sbytes);
        const int row0 = ti.b * p.Lmax + ti.t * kTok;
#pragma unroll
        for (int j = 0; j < 8; ++j) tma_load_2d(dst + j * kBlk, &tm_c, &bar[B_FULL + st], j * 64, row0);
        if (rank == 0) tma_load_2d(dst + 8 * kBlk, &tm_kr, &bar[B_FULL + st], 0, row0);
        last_use[st] = ti.i;
        return true;
      });
      for (int s = 0; s < kStages; ++s)  // let every issued copy land before the CTA winds down
        if (last_use[s] >= 0) mbar_wait_drain(&bar[B_FULL + s], (uint32_t)(last_use[s] / kStages) & 1u, wc);
    }
  } else if (run && warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      if (rank == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, kTok, 0, 0);
        for_each_tile(p, g, [&](const TileInfo& ti) {
          const int st = ti.i % kStages, slot = ti.i & 1;
          const uint32_t ph = (uint32_t)(ti.i / kStages) & 1u, sph = (uint32_t)(ti.i >> 1) & 1u;
          if (!mbar_wait(&bar[B_FULL + st], ph, wc)) return false;
          if (!mbar_wait(&bar[B_SEMPTY + slot], sph ^ 1u, wc)) return false;
          if (ti.first && !mbar_wait(&bar[B_QREADY], (uint32_t)ti.k & 1u, wc)) return false;
          tc_fence_after();
          const uint32_t sbase = smem_u32(smem + st * kStage0);
          const uint32_t d = tmem + (uint32_t)slot * kTok;
#pragma unroll 4
          for (int kk = 0; kk < 36; ++kk) {  // K = 576 in steps of 16
            const uint64_t bd = smem_desc(sbase + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024, 2);
            mma_ts(d, tmem + kQCol + (uint32_t)kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar[B_SFULL + slot]);
          mma_commit(&bar[B_EMPTY + st]);
          return true;
        });
      } else {
        constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
        for_each_tile(p, g, [&](const TileInfo& ti) {
          const int st = ti.i % kStages, slot = ti.i & 1;
          const uint32_t ph = (uint32_t)(ti.i / kStages) & 1u, sph = (uint32_t)(ti.i >> 1) & 1u;
          if (!mbar_wait(&bar[B_FULL + st], ph, wc)) return false;
          if (!mbar_wait(&bar[B_PREADY + slot], sph, wc)) return false;
          if (ti.first && ti.k > 0 && !mbar_wait(&bar[B_OFREE], (uint32_t)(ti.k - 1) & 1u, wc))
            return false;
          fence_proxy_async_cta();  // P arrived through the generic proxy; the MMA reads it
          tc_fence_after();
          const int nvt = min(ti.L - ti.t * kTok, kTok);
          const int nk = (nvt + 15) >> 4;
          const uint32_t sbase = smem_u32(smem + st * kStage1);
          const uint32_t pbase = smem_u32(smem + kOffP + slot * kPBytes);
          for (int kt = 0; kt < nk; ++kt) {  // K = tokens in steps of 16
            const uint64_t ad = smem_desc(pbase + kt * 32, 16, 1024, 2);
#pragma unroll
            for (int n = 0; n < 2; ++n) {   // N = 512 latent columns as 2 x 256
              const uint64_t bd = smem_desc(sbase + n * 4 * kBlk + kt * 2048, kBlk, 1024, 2);
              mma_ss(tmem + (uint32_t)n * 256, ad, bd, idesc, (kt > 0 || !ti.first) ? 1u : 0u);
            }
          }
          mma_commit(&bar[B_PVDONE + slot]);
          mma_commit(&bar[B_EMPTY + st]);
          return true;
        });
      }
      mma_commit(&bar[B_DRAIN]);  // every MMA has finished before tensor memory is released
      mbar_wait_drain(&bar[B_DRAIN], 0, wc);
    }
  } else if (run && warp == 2) {
    // ------------------------------------------------ value CTA: P-slot releaser
    if (rank == 1 && lane == 0) {
      for_each_tile(p, g, [&](const TileInfo& ti) {
        const int slot = ti.i & 1;
        if (!mbar_wait(&bar[B_PVDONE + slot], (uint32_t)(ti.i >> 1) & 1u, wc)) return false;
        mbar_arrive_remote(&bar[B_PEMPTY + slot], 0);
        return true;
      });
    }
  } else if (run) {
    // ------------------------------------------------ warps 3..6: one row per thread
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int SH = p.S * p.H;
    const int gr = rb * 128 + r;
    const bool valid = gr < SH;
    const int s_r = valid ? gr / p.H : 0, h_r = valid ? gr - (gr / p.H) * p.H : 0;

    if (rank == 0) {
      // ---------------------------------------- scores + online softmax
      const uint32_t p_remote = map_to_cta(smem_u32(smem + kOffP), 1);
      const uint32_t a_remote = map_to_cta(smem_u32(smem + kOffAlpha), 1);
      const uint32_t pfull_remote = map_to_cta(smem_u32(&bar[B_PFULL]), 1);
      float m_ref = -INFINITY, l = 0.f;
      int limit = 0;
      for_each_tile(p, g, [&](const TileInfo& ti) {
        if (ti.first) {  // the previous segment's MMAs are done: load this segment's Q
          limit = valid ? ti.L - p.S + s_r + 1 : 0;
          const uint4* qrow = reinterpret_cast<const uint4*>(
              p.q_cat + (((size_t)ti.b * p.S + s_r) * p.H + h_r) * 576);
#pragma unroll 1
          for (int c3 = 0; c3 < 9; c3 += 3) {  // 3 x 3 chunks: 24 loads in flight per thread
            uint32_t v[3][32];
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const uint4 x = valid ? __ldg(qrow + (c3 + c) * 8 + u) : make_uint4(0, 0, 0, 0);
                v[c][4 * u] = x.x; v[c][4 * u + 1] = x.y; v[c][4 * u + 2] = x.z; v[c][4 * u + 3] = x.w;
              }
#pragma unroll
            for (int c = 0; c < 3; ++c) tmem_st32(tl + kQCol + (uint32_t)(c3 + c) * 32, v[c]);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar[B_QREADY]);
          m_ref = -INFINITY;
          l = 0.f;
        }
        const int slot = ti.i & 1;
        const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u;
        if (!warp_wait(&bar[B_SFULL + slot], sph, wc)) return false;
        tc_fence_after();
        uint32_t sv[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tmem_ld32(tl + (uint32_t)slot * kTok, lo);
          tmem_ld32(tl + (uint32_t)slot * kTok + 32, hi);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar[B_SEMPTY + slot]);

        const int nv = min(max(limit - ti.t * kTok, 0), kTok);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTok; ++c) {
          const float s2 = __uint_as_float(sv[c]) * p.scale_log2;
          sv[c] = __float_as_uint(s2);
          if (c < nv) mx = fmaxf(mx, s2);
        }
        float alpha = 1.f;
        if (mx > m_ref + 8.f) {
          const float mn = ceilf(mx);
          alpha = (m_ref == -INFINITY) ? 0.f : exp2_int((int)(m_ref - mn));
          l *= alpha;
          m_ref = mn;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float e0 = (2 * c < nv) ? exp2f(__uint_as_float(sv[2 * c]) - mu) : 0.f;
          const float e1 = (2 * c + 1 < nv) ? exp2f(__uint_as_float(sv[2 * c + 1]) - mu) : 0.f;
          pk[c] = pack_bf16x2(e0, e1);
          const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[c]);
          lsum += __low2float(b2) + __high2float(b2);
        }
        l += lsum;

        if (!warp_wait(&bar[B_PEMPTY + slot], sph ^ 1u, wc)) return false;
        const uint32_t row = p_remote + (uint32_t)slot * kPBytes + (uint32_t)r * 128;
        const uint32_t rbar = pfull_remote + (uint32_t)slot * 8;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)  // 128-byte swizzle: chunk ch of row r sits at ch ^ (r & 7)
          st_async_v4(row + (uint32_t)((ch ^ (r & 7)) << 4),
                      make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]), rbar);
        st_async_f32(a_remote + (uint32_t)(slot * 128 + r) * 4, alpha, rbar);
        if (ti.last && valid) p.ml[((size_t)ti.slot * p.n_rb + rb) * 128 + r] = make_float2(mu, l);
        return true;
      });
    } else {
      // ---------------------------------------- rescale, tail zeroing, epilogue
      const int wt = threadIdx.x - 96;  // 0..127
      const volatile float* alpha_buf = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
      for_each_tile(p, g, [&](const TileInfo& ti) {
        const int slot = ti.i & 1, st = ti.i % kStages;
        const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u, ph = (uint32_t)(ti.i / kStages) & 1u;
        if (!warp_wait(&bar[B_PFULL + slot], sph, wc)) return false;
        const float alpha = alpha_buf[slot * 128 + r];
        if (wt == 0) mbar_arrive_expect_tx(&bar[B_PFULL + slot], kPTx);  // arm the slot's next phase
        const bool need = !ti.first && alpha != 1.f;
        if (__any_sync(0xffffffffu, need)) {
          // O rows change only after the previous tile's P . C has completed
          if (!warp_wait(&bar[B_PVDONE + (slot ^ 1)], (uint32_t)((ti.i - 1) >> 1) & 1u, wc)) return false;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 16; ++c) {
            uint32_t v[32];
            tmem_ld32(tl + (uint32_t)c * 32, v);
            tmem_wait_ld();
            if (need) {
#pragma unroll
              for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * alpha);
            }
            tmem_st32(tl + (uint32_t)c * 32, v);
          }
          tmem_wait_st();
        }
        const int nvt = min(ti.L - ti.t * kTok, kTok);
        if (nvt & 15) {
          // cache rows past the sequence end inside the last 16-row MMA step hold
          // arbitrary bytes; their weights are 0 but 0 * NaN is not, so zero them
          if (!warp_wait(&bar[B_FULL + st], ph, wc)) return false;
          const int z0 = nvt, nzr = ((nvt + 15) & ~15) - nvt;
          uint8_t* sb = smem + st * kStage1;
          for (int idx = wt; idx < nzr * 64; idx += 128) {
            const int blk = idx / (nzr * 8), rem = idx - blk * (nzr * 8);
            *reinterpret_cast<uint4*>(sb + blk * kBlk + (z0 + (rem >> 3)) * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_cta();
        }
        tc_fence_before();
        mbar_arrive(&bar[B_PREADY + slot]);
        if (ti.last) {
          if (!warp_wait(&bar[B_PVDONE + slot], sph, wc)) return false;
          tc_fence_after();
          // column-major [512][128]: for each column a warp stores 32 consecutive floats
          float* dst = p.opart + ((size_t)ti.slot * p.n_rb + rb) * 512 * 128 + r;
#pragma unroll 1
          for (int c = 0; c < 16; ++c) {
            uint32_t v[32];
            tmem_ld32(tl + (uint32_t)c * 32, v);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
              for (int u = 0; u < 32; ++u) dst[(size_t)(c * 32 + u) * 128] = __uint_as_float(v[u]);
            }
          }
          tc_fence_before();
          mbar_arrive(&bar[B_OFREE]);
        }
        return true;
      });
    }
  }

  // ------------------------------------------------ wind down
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  cluster_sync();
}

}  // namespace mla
