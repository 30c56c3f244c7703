// prefill.cuh -- causal attention of many query positions per sequence
// (prefill and long chunks), in the expanded form.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention":
//   KeyValue:  k^C_{t,i} = W_i^UK c_t,  v^C_{t,i} = W_i^UV c_t,  k^R_t = RoPE_t(.)
//   Query:     q_{t,i} = [q^C_{t,i}; q^R_{t,i}]  (q^R rotated at t)
//   注意力计算: o_{t,i} = sum_{j <= t} softmax_j(q_{t,i} . [k^C_{j,i}; k^R_j] / sqrt(192)) v^C_{j,i}
// When every position of a prompt queries the cache, expanding the keys and
// values once per head (mla_prefill_expand: 2 x 128 x 512 x 2 flops per token
// and head) makes each (query, key, head) cost 2 x (192 + 128) flops, where the
// absorbed form of "潜在向量的作用" costs 2 x (576 + 512).
//
// A work item is 128 consecutive query positions of one (sequence, head); its
// rows see keys 0 .. their own position, so the item walks key tiles of 128
// from the start of the sequence to the tile holding its last position.  A
// unit pairs a head's last query block with its first, its second last with
// its second, and so on, so that the units of a sequence cost the same; one
// persistent CTA per SM takes units round-robin, head after head, so that the
// CTAs work on a few heads at a time and a head's expanded keys and values
// are read from HBM about once and then from L2.
//
// Per CTA (384 threads): warp 0 issues the TMA copies of Q (once per item:
// q^C and q^R as three 128-byte-swizzle atoms) and of each key tile (k^C,
// k^R), warp 2 those of each value tile (v^C); one thread of warp 1 issues
// the QK^T MMAs and one of warp 3 the P.V MMAs; warps 4..11 run the online
// softmax and the epilogue, two threads per row (one per 64-column half of
// the scores and of O).
// Tensor memory holds three 128-column score buffers S and the 128 x 128 fp32
// output O (columns 384..511).  QK^T runs up to three tiles ahead of P.V; the
// softmax writes P (bf16) over the first half of each 64-column half of its
// S buffer and P.V reads it from there (A operand in tensor memory).  The online softmax keeps an integer reference exponent per
// row (log2 units) that moves only when a tile's maximum passes it by more
// than 8, so every rescale of O and of the row sum is an exact power of two.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kPfThreads = 384;
constexpr int kPfAtom = 128 * 128;  // 128 rows x 64 bf16 columns (one swizzle atom column), 16 KB
constexpr int kPfQ = 3 * kPfAtom;   // q^C (two atoms) + q^R (one)
constexpr int kPfK = 3 * kPfAtom;   // k^C (two atoms) + k^R (one)
constexpr int kPfV = 2 * kPfAtom;   // v^C (two atoms)
constexpr int kPfKStages = 2, kPfVStages = 2;
static_assert(kPfKStages == 2 && kPfVStages == 2, "the producers index two-deep rings");
constexpr int kPfOffK = kPfQ;
constexpr int kPfOffV = kPfOffK + kPfKStages * kPfK;
constexpr int kPfOffBar = kPfOffV + kPfVStages * kPfV;
enum : int {
  PF_QFULL = 0, PF_QEMPTY = 1, PF_KFULL = 2, PF_KEMPTY = 4, PF_VFULL = 6, PF_VEMPTY = 8,
  PF_SFULL = 10, PF_PREADY = 13, PF_PVDONE = 16, PF_OFREE = 19, PF_DRAIN = 20,
  PF_XCH = 21,   // row-maximum exchange of a row's two threads [tile parity][quadrant]
  PF_XL = 29,    // row-sum exchange at an item's end [quadrant]
  PF_DRAIN2 = 33,  // the P.V issuer's final drain
  PF_NBARS = 34
};
// the two threads of a row exchange partial row maxima [tile parity][half][row]
// and, at an item's end, partial row sums [half][row]
constexpr int kPfOffXch = kPfOffBar + PF_NBARS * 8 + 16;
constexpr int kPfXchBytes = 2 * 2 * 128 * 4 + 2 * 128 * 4;
constexpr size_t kPfSmem = (size_t)kPfOffXch + kPfXchBytes;
static_assert(kPfSmem <= 232448, "prefill shared memory exceeds 227 KB");
constexpr uint32_t kPfOCol = 384;  // O; the score buffers sit at columns 0, 128 and 256

struct PrefillParams {
  __nv_bfloat16* out;        // [B, S, H, 128]
  const int32_t* seqlens;    // [B]: cached tokens, the S new ones included
  int B, S, H, Lmax;
  int nq;                    // query blocks of 128 per (sequence, head)
  int n_units;               // B * H * ceil(nq / 2)
  float scale_log2;          // softmax scale * log2(e)
  uint32_t* status;
  uint64_t timeout_ns;
  unsigned long long* trace;  // timeline of a diagnostic build (MLA_PREFILL_TRACE), else unused
};

// Diagnostic timeline: with MLA_PREFILL_TRACE defined, CTAs 0..7 stamp
// %globaltimer at events of their first 128 key tiles into
// trace[cta][event][tile].  Compiled out otherwise.
enum : int {
  PT_KFULL = 0, PT_QK = 1, PT_SREADY = 2, PT_PREADY = 3, PT_PSEEN = 4, PT_VFULL = 5, PT_PV = 6, PT_KISSUE = 7,
  PT_NEV = 8
};
#ifdef MLA_PREFILL_TRACE
#define PF_TRACE(p, ev, g)                                                                   \
  do {                                                                                       \
    if ((p).trace && blockIdx.x < 8 && (g) < 128)                                            \
      (p).trace[((size_t)blockIdx.x * PT_NEV + (ev)) * 128 + (g)] = global_timer_ns();       \
  } while (0)
#else
#define PF_TRACE(p, ev, g) \
  do {                     \
  } while (0)
#endif

struct PfItem {
  int b, h, s0, nrow, p0, p_last, nt;
  bool ok;
};

// Work unit u of (sequence, head) bh = u / np: query blocks nq - 1 - k and k
// (k = u mod np, np = ceil(nq / 2); one block when they coincide), so that
// every unit of a sequence walks the same number of key tiles and the CTAs,
// taking units round-robin, stay on the same few heads (whose expanded keys
// and values then come from L2).
__device__ __forceinline__ int pf_unit_blocks(const PrefillParams& p, int u, int (&qb)[2], int& bh) {
  const int np = (p.nq + 1) >> 1;
  bh = u / np;
  const int k = u - bh * np;
  qb[0] = p.nq - 1 - k;
  qb[1] = k;
  return qb[0] == k ? 1 : 2;
}

__device__ __forceinline__ PfItem pf_item(const PrefillParams& p, int bh, int qb) {
  PfItem it;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  const int L = __ldg(p.seqlens + it.b);
  it.ok = L >= p.S && L <= p.Lmax;
  it.s0 = qb * 128;
  it.nrow = min(128, p.S - it.s0);
  it.p0 = L - p.S + it.s0;            // position of the block's first query
  it.p_last = it.p0 + it.nrow - 1;    // and of its last (at most L - 1)
  it.nt = it.ok ? it.p_last / 128 + 1 : 0;
  return it;
}

// This CTA's items in order: units blockIdx.x, blockIdx.x + gridDim.x, ...,
// each one or two query blocks.
struct PfIter {
  int u = (int)blockIdx.x, slot = 0;
  __device__ __forceinline__ bool next(const PrefillParams& p, PfItem& it) {
    while (u < p.n_units) {
      int qb[2], bh;
      const int n = pf_unit_blocks(p, u, qb, bh);
      if (slot < n) {
        it = pf_item(p, bh, qb[slot++]);
        return true;
      }
      u += (int)gridDim.x;
      slot = 0;
    }
    return false;
  }
};

__device__ __forceinline__ bool pf_warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// Exact 2^d for an integer d <= 0 (0 below the normal range).
__device__ __forceinline__ float pf_exp2_int(int d) {
  return d <= -127 ? 0.f : __int_as_float((127 + d) << 23);
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qr,
                   const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_kr,
                   const __grid_constant__ CUtensorMap tm_vc, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPfOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + PF_NBARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < PF_NBARS; ++i) {
      uint32_t n = 1;  // TMA arrivals and MMA commits
      if ((i >= PF_PREADY && i < PF_PREADY + 3) || i == PF_OFREE) n = 256;  // every row thread
      if (i >= PF_XCH && i < PF_DRAIN2) n = 64;                             // the two warps of a quadrant
      mbar_init(&bar[i], n);
    }
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_qn);
    tma_prefetch_desc(&tm_qr);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_kr);
    tma_prefetch_desc(&tm_vc);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // q, the expanded keys and values and the cache come from earlier kernels

  if (warp == 0 || warp == 2) {
    if (lane == 0) {
      // -------------------------------------------------- TMA producers: warp 0
      // loads Q and the key tiles, warp 2 the value tiles, each on its own ring
      // so that neither waits for the other's slots
      const bool keys = warp == 0;
      uint32_t c = 0, it = 0, q_issued = 0;
      bool ok = true;
      PfIter iter;
      PfItem ii;
      while (ok && iter.next(p, ii)) {
        if (!ii.ok) {
          if (keys) atomicOr(p.status, kDevErrBadSeqlen);
          continue;
        }
        if (keys) {
          if (it > 0 && !mbar_wait(&bar[PF_QEMPTY], (it - 1) & 1u, wc)) break;
          const int qrow = ii.b * p.S + ii.s0;
          mbar_arrive_expect_tx(&bar[PF_QFULL], (uint32_t)kPfQ);
          tma_load_4d(smem, &tm_qn, &bar[PF_QFULL], 0, qrow, 0, ii.h);
          tma_load_3d(smem + 2 * kPfAtom, &tm_qr, &bar[PF_QFULL], 0, qrow, ii.h);
          q_issued = it + 1;
        }
        const int krow0 = ii.b * p.Lmax;
        for (int t = 0; t < ii.nt; ++t, ++c) {
          const int krow = krow0 + t * 128;
          const uint32_t st = c % 2;  // both rings are two deep
          if (c >= 2 && !mbar_wait(&bar[(keys ? PF_KEMPTY : PF_VEMPTY) + st], ((c / 2) - 1) & 1u, wc)) {
            ok = false;
            break;
          }
          if (keys) {
            PF_TRACE(p, PT_KISSUE, c);
            uint8_t* kb = smem + kPfOffK + st * kPfK;
            mbar_arrive_expect_tx(&bar[PF_KFULL + st], (uint32_t)kPfK);
            tma_load_4d(kb, &tm_kc, &bar[PF_KFULL + st], 0, krow, 0, ii.h);
            tma_load_2d(kb + 2 * kPfAtom, &tm_kr, &bar[PF_KFULL + st], 0, krow);
          } else {
            mbar_arrive_expect_tx(&bar[PF_VFULL + st], (uint32_t)kPfV);
            tma_load_4d(smem + kPfOffV + st * kPfV, &tm_vc, &bar[PF_VFULL + st], 0, krow, 0, ii.h);
          }
        }
        ++it;
      }
      // every copy issued lands before the CTA winds down
      const int full = keys ? PF_KFULL : PF_VFULL;
      for (uint32_t j = c > 2u ? c - 2 : 0; j < c; ++j) mbar_wait_drain(&bar[full + j % 2], (j / 2) & 1u, wc);
      if (q_issued > 0) mbar_wait_drain(&bar[PF_QFULL], (q_issued - 1) & 1u, wc);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------ QK^T issuer
      // Two threads issue the MMAs, each with its own commits: this one QK^T,
      // warp 3's P.V (they write different tensor-memory columns, and the
      // barriers order them), so neither waits behind the other's issue.
      constexpr uint32_t idq = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
      uint32_t kc = 0, g = 0, it = 0;
      bool ok = true;
      PfIter iter;
      PfItem ii;
      while (ok && iter.next(p, ii)) {
        if (!ii.ok) continue;
        if (!mbar_wait(&bar[PF_QFULL], it & 1u, wc)) break;
        for (int t = 0; t < ii.nt; ++t, ++g) {
          // QK^T of tile g into score buffer g % 3, whose previous P (tile
          // g - 3) must have been consumed by its P.V
          const uint32_t sb = g % 3, st = kc % kPfKStages;
          if ((g >= 3 && !mbar_wait(&bar[PF_PVDONE + sb], ((g / 3) - 1) & 1u, wc)) ||
              !mbar_wait(&bar[PF_KFULL + st], (kc / kPfKStages) & 1u, wc)) {
            ok = false;
            break;
          }
          PF_TRACE(p, PT_KFULL, g);
          tc_fence_after();
          // descriptors built once and stepped (a descriptor's start address is
          // its low field, in 16-byte units, and stays below 2^14 here)
          const uint64_t qd = smem_desc(smem_u32(smem), 16, 1024, 2);
          const uint64_t kd = smem_desc(smem_u32(smem + kPfOffK + st * kPfK), 16, 1024, 2);
          const uint32_t sd = tmem + sb * 128;
#pragma unroll
          for (int kk = 0; kk < 12; ++kk) {  // 192 = 3 atoms x 4 K-steps of 16
            const uint64_t off = (uint64_t)(((kk >> 2) * kPfAtom + (kk & 3) * 32) >> 4);
            mma_ss(sd, qd + off, kd + off, idq, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar[PF_KEMPTY + st]);
          mma_commit(&bar[PF_SFULL + sb]);
          PF_TRACE(p, PT_QK, g);
          ++kc;
        }
        if (!ok) break;
        mma_commit(&bar[PF_QEMPTY]);  // Q is free once the item's QK^T are done
        ++it;
      }
      mma_commit(&bar[PF_DRAIN]);  // every MMA of this thread has finished before tensor memory is released
      mbar_wait_drain(&bar[PF_DRAIN], 0, wc);
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // -------------------------------------------------------- P.V issuer
      constexpr uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);  // O += P V, V MN-major
      uint32_t vc = 0, g = 0, it = 0;
      bool ok = true;
      PfIter iter;
      PfItem ii;
      while (ok && iter.next(p, ii)) {
        if (!ii.ok) continue;
        for (int t = 0; t < ii.nt; ++t) {
          const uint32_t sb = g % 3, st = vc % kPfVStages;
          if (!mbar_wait(&bar[PF_PREADY + sb], (g / 3) & 1u, wc) ||
              (t == 0 && it > 0 && !mbar_wait(&bar[PF_OFREE], (it - 1) & 1u, wc))) {
            ok = false;
            break;
          }
          PF_TRACE(p, PT_PSEEN, g);
          if (!mbar_wait(&bar[PF_VFULL + st], (vc / kPfVStages) & 1u, wc)) {
            ok = false;
            break;
          }
          PF_TRACE(p, PT_VFULL, g);
          tc_fence_after();
          // tokens any row of the block sees in this tile; rows past them are
          // weighted 0, but 0 * NaN is not 0, so the rows up to the next
          // multiple of 16 (one MMA K-step) are zeroed
          const int nvt = min(128, ii.p_last + 1 - t * 128);
          const int nk = (nvt + 15) >> 4;
          uint8_t* vb = smem + kPfOffV + st * kPfV;
          if (nvt & 15) {
            for (int a = 0; a < 2; ++a)
              for (int row = nvt; row < nk * 16; ++row)
                for (int ch = 0; ch < 8; ++ch)
                  *reinterpret_cast<uint4*>(vb + a * kPfAtom + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_cta();
          }
          const uint64_t vd = smem_desc(smem_u32(vb), kPfAtom, 1024, 2);
          const uint32_t pa = tmem + sb * 128, od = tmem + kPfOCol, acc0 = t > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // up to 8 K-steps of 16 keys: 2048 bytes of V each
            if (kk < nk)
              mma_ts(od, pa + (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8), vd + (uint64_t)(kk * 128), idv,
                     kk > 0 ? 1u : acc0);
          mma_commit(&bar[PF_VEMPTY + st]);
          mma_commit(&bar[PF_PVDONE + sb]);
          PF_TRACE(p, PT_PV, g);
          ++vc;
          ++g;
        }
        ++it;
      }
      mma_commit(&bar[PF_DRAIN2]);  // every MMA of this thread has finished before tensor memory is released
      mbar_wait_drain(&bar[PF_DRAIN2], 0, wc);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax + epilogue
    // Two threads per row (warps 4..7: score columns 0..63, warps 8..11:
    // 64..127, of the rows of tensor-memory quadrant warp & 3).  They
    // exchange partial row maxima per tile and partial row sums per item
    // through shared memory and mbarriers, so both take the same reference
    // exponent; each rescales and writes its own 64 columns of O.
    const int q4 = warp & 3, hw = (warp - 4) >> 2;
    const int r = q4 * 32 + lane;  // this thread's row = tensor-memory lane
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    float* xmax = reinterpret_cast<float*>(smem + kPfOffXch);  // [parity][half][row]
    float* xsum = xmax + 2 * 2 * 128;                          // [half][row]
    uint32_t g = 0, it = 0;
    bool ok = true;
    PfIter iter;
    PfItem ii;
    while (ok && iter.next(p, ii)) {
      if (!ii.ok) continue;
      const int pr = min(ii.p0 + r, ii.p_last);  // rows past the block's last query repeat it
      float m_ref = -INFINITY, l = 0.f;
      for (int t = 0; t < ii.nt; ++t) {
        const uint32_t sb = g % 3, par = g & 1u;
        if (!pf_warp_wait(&bar[PF_SFULL + sb], (g / 3) & 1u, wc)) {
          ok = false;
          break;
        }
        if (r == 0 && hw == 0) PF_TRACE(p, PT_SREADY, g);
        tc_fence_after();
        const uint32_t sc = tl + sb * 128 + (uint32_t)(hw * 64);
        // visible columns of this thread's half
        const int nv = min(max(pr + 1 - t * 128 - hw * 64, 0), 64);
        uint32_t v[64];
        tmem_ld32(sc, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(sc + 32u, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_wait_ld();
        const bool full = __all_sync(0xffffffffu, nv == 64);  // no column of this warp's half is masked
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = -INFINITY;
        if (full) {
#pragma unroll
          for (int u = 0; u < 64; ++u) pm[u & 7] = fmaxf(pm[u & 7], __uint_as_float(v[u]));
        } else {
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u < nv) pm[u & 7] = fmaxf(pm[u & 7], __uint_as_float(v[u]));
        }
        float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        // the row's maximum over both halves
        xmax[(par * 2 + hw) * 128 + r] = mx;
        mbar_arrive(&bar[PF_XCH + par * 4 + q4]);
        if (!mbar_wait(&bar[PF_XCH + par * 4 + q4], (g >> 1) & 1u, wc)) {
          ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xmax[(par * 2 + (hw ^ 1)) * 128 + r]) * p.scale_log2;
        const float cm = ceilf(mx);
        int ex = 0;  // O and l are rescaled by 2^-ex; 255 stands for 0
        if (cm > m_ref + 8.f) {
          ex = (m_ref == -INFINITY) ? 255 : (int)fminf(cm - m_ref, 255.f);
          l = (ex == 255) ? 0.f : l * pf_exp2_int(-ex);
          m_ref = cm;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        const bool need = t > 0 && ex != 0;
        if (__any_sync(0xffffffffu, need)) {
          // O holds this item's earlier tiles once the previous P.V has completed
          if (!pf_warp_wait(&bar[PF_PVDONE + (g - 1) % 3], ((g - 1) / 3) & 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = ex == 255 ? 0.f : pf_exp2_int(-ex);
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            const uint32_t a = tl + kPfOCol + (uint32_t)(hw * 64 + c * 32);
            tmem_ld32(a, o);
            tmem_wait_ld();
            if (need) {
#pragma unroll
              for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            }
            tmem_st32(a, o);
          }
        }
        // P = 2^(s scale log2 e - m) in bf16, written over the first 32
        // columns of this thread's 64-column half (already read above)
        float lsa[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) lsa[k] = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          float e0 = ex2_approx(fmaf(__uint_as_float(v[2 * u]), p.scale_log2, -mu));
          float e1 = ex2_approx(fmaf(__uint_as_float(v[2 * u + 1]), p.scale_log2, -mu));
          if (!full) {
            e0 = 2 * u < nv ? e0 : 0.f;
            e1 = 2 * u + 1 < nv ? e1 : 0.f;
          }
          pk[u] = pack_bf16x2(e0, e1);
          // the row sum adds exactly the bf16 weights that P.V multiplies
          lsa[(2 * u) & 7] += __uint_as_float(pk[u] << 16);
          lsa[(2 * u + 1) & 7] += __uint_as_float(pk[u] & 0xffff0000u);
        }
        tmem_st32(sc, pk);
        const float ls = ((lsa[0] + lsa[1]) + (lsa[2] + lsa[3])) + ((lsa[4] + lsa[5]) + (lsa[6] + lsa[7]));
        tmem_wait_st();
        l += ls;
        tc_fence_before();
        mbar_arrive(&bar[PF_PREADY + sb]);
        if (r == 0 && hw == 0) PF_TRACE(p, PT_PREADY, g);
        ++g;
      }
      if (!ok) break;
      // epilogue: out = O / l once the item's last P.V has completed, l the
      // sum of both halves' partial sums
      xsum[hw * 128 + r] = l;
      mbar_arrive(&bar[PF_XL + q4]);
      if (!pf_warp_wait(&bar[PF_XL + q4], it & 1u, wc)) break;
      l += xsum[(hw ^ 1) * 128 + r];
      if (!pf_warp_wait(&bar[PF_PVDONE + (g - 1) % 3], ((g - 1) / 3) & 1u, wc)) break;
      tc_fence_after();
      const float inv = 1.f / l;
      const bool valid = r < ii.nrow;
      uint4* orow = reinterpret_cast<uint4*>(p.out + (((size_t)ii.b * p.S + ii.s0 + r) * p.H + ii.h) * 128 + hw * 64);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + kPfOCol + (uint32_t)(hw * 64 + c * 32), v);
        tmem_wait_ld();
        uint32_t o[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          o[u] = pack_bf16x2(__uint_as_float(v[2 * u]) * inv, __uint_as_float(v[2 * u + 1]) * inv);
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) orow[c * 4 + u] = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar[PF_OFREE]);
      ++it;
    }
  }

  // ---------------------------------------------------------------- wind down
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace mla
