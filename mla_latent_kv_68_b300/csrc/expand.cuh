// expand.cuh -- the keys and values of every cached token expanded per head,
// for the prefill's attention over them.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / KeyValue":
//   k^C_{t,i} = W_i^UK c_t,   v^C_{t,i} = W_i^UV c_t,   W_i in R^{128 x 512}.
// For T cached tokens and H heads that is a [T x 512] x [512 x 2 H 128] GEMM
// whose output (T x 2 H x 128 bf16) is as large as both inputs together
// many times over, so every byte of it is written once and the inputs are
// re-read from L2.
//
// One persistent CTA per SM takes units of (128 tokens, up to kExGroup heads of
// one weight) in turn.  The unit's 128 x 512 latent rows stay in shared memory
// (A operand, eight 128-byte-swizzle atoms, K-major) while the heads' weight
// rows stream through a ring of 32 KB boxes (128 rows x two atoms; B operand,
// K-major).  Per head, sixteen MMAs of M = 128 tokens, N = 128 outputs, K = 16
// accumulate in one of four tensor-memory buffers; four epilogue warps turn a
// finished buffer into bf16 rows (one token per thread, 256 contiguous bytes
// per head) while the MMAs of the next heads run.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kExThreads = 256;   // warp 0 TMA, warp 1 MMA, warps 4..7 epilogue
constexpr int kExAtom = 128 * 128;
constexpr int kExA = 8 * kExAtom;  // 128 tokens x 512 latent columns
constexpr int kExB = 2 * kExAtom;  // 128 weight rows x 128 columns
constexpr int kExStages = 3;
constexpr int kExGroup = 16;       // heads per unit
constexpr int kExOffB = kExA;
constexpr int kExOffBar = kExOffB + kExStages * kExB;
enum : int {
  EX_AFULL = 0, EX_AEMPTY = 1, EX_BFULL = 2, EX_BEMPTY = 2 + kExStages, EX_DFULL = 2 + 2 * kExStages,
  EX_DEMPTY = EX_DFULL + 4, EX_DRAIN = EX_DEMPTY + 4, EX_NBARS = EX_DRAIN + 1
};
constexpr size_t kExSmem = (size_t)kExOffBar + EX_NBARS * 8 + 16;

struct ExpandParams {
  __nv_bfloat16* k_c;   // [T][H][128]
  __nv_bfloat16* v_c;   // [T][H][128]
  int T, H;
  int n_tt, n_grp;      // token tiles of 128; head groups per tile (over 2 H heads: W_UK's, then W_UV's)
  uint32_t* status;
  uint64_t timeout_ns;
};

// Unit u: token tile u / n_grp, heads [j0, j1) of the 2 H (k heads, then v heads).
struct ExUnit {
  int row0, j0, j1;
};
__device__ __forceinline__ ExUnit ex_unit(const ExpandParams& p, int u) {
  ExUnit e;
  const int tt = u / p.n_grp, gi = u - tt * p.n_grp;
  e.row0 = tt * 128;
  // groups never straddle the two weights: n_grp / 2 groups per weight
  const int per_w = p.n_grp / 2, w = gi / per_w, gw = gi - w * per_w;
  e.j0 = w * p.H + gw * kExGroup;
  e.j1 = w * p.H + min(p.H, (gw + 1) * kExGroup);
  return e;
}

__global__ void __launch_bounds__(kExThreads, 1)
    expand_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_wv, const ExpandParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kExOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + EX_NBARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const int n_units = p.n_tt * p.n_grp;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < EX_NBARS; ++i) mbar_init(&bar[i], (i >= EX_DEMPTY && i < EX_DEMPTY + 4) ? 128u : 1u);
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_wk);
    tma_prefetch_desc(&tm_wv);
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
  pdl_wait();  // the cache rows may come from the kernel before this one

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t bc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++uc) {
        const ExUnit e = ex_unit(p, u);
        if (uc > 0 && !mbar_wait(&bar[EX_AEMPTY], (uc - 1) & 1u, wc)) break;
        mbar_arrive_expect_tx(&bar[EX_AFULL], (uint32_t)kExA);
        tma_load_3d(smem, &tm_c, &bar[EX_AFULL], 0, e.row0, 0);
        tma_load_3d(smem + 4 * kExAtom, &tm_c, &bar[EX_AFULL], 0, e.row0, 4);
        for (int j = e.j0; ok && j < e.j1; ++j) {
          const CUtensorMap* tw = j < p.H ? &tm_wk : &tm_wv;
          const int wrow = (j < p.H ? j : j - p.H) * 128;
          for (int ks = 0; ks < 4; ++ks, ++bc) {
            const uint32_t st = bc % kExStages;
            if (bc >= (uint32_t)kExStages &&
                !mbar_wait(&bar[EX_BEMPTY + st], ((bc / kExStages) - 1) & 1u, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bar[EX_BFULL + st], (uint32_t)kExB);
            tma_load_3d(smem + kExOffB + st * kExB, tw, &bar[EX_BFULL + st], 0, wrow, ks * 2);
          }
        }
      }
      for (uint32_t j = bc > (uint32_t)kExStages ? bc - kExStages : 0; j < bc; ++j)
        mbar_wait_drain(&bar[EX_BFULL + j % kExStages], (j / kExStages) & 1u, wc);
      if (uc > 0) mbar_wait_drain(&bar[EX_AFULL], (uc - 1) & 1u, wc);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
      uint32_t bc = 0, uc = 0, e = 0;  // weight stages, units, accumulator uses
      bool ok = true;
      const uint32_t a0 = smem_u32(smem);
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++uc) {
        const ExUnit un = ex_unit(p, u);
        if (!mbar_wait(&bar[EX_AFULL], uc & 1u, wc)) break;
        for (int j = un.j0; ok && j < un.j1; ++j, ++e) {
          const uint32_t buf = e % 4;
          if (e >= 4 && !mbar_wait(&bar[EX_DEMPTY + buf], ((e / 4) - 1) & 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int ks = 0; ks < 4; ++ks, ++bc) {
            const uint32_t st = bc % kExStages;
            if (!mbar_wait(&bar[EX_BFULL + st], (bc / kExStages) & 1u, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors built once and stepped (the start address is the low
            // field, in 16-byte units; every address here is below 2^18)
            const uint64_t bd = smem_desc(smem_u32(smem + kExOffB + st * kExB), 16, 1024, 2);
            const uint64_t ad = smem_desc(a0 + (uint32_t)(ks * 2 * kExAtom), 16, 1024, 2);
            const uint32_t dd = tmem + buf * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // two atoms x four K-steps of 16
              const uint64_t off = (uint64_t)((((kk >> 2) * kExAtom) + (kk & 3) * 32) >> 4);
              mma_ss(dd, ad + off, bd + off, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bar[EX_BEMPTY + st]);
          }
          if (ok) mma_commit(&bar[EX_DFULL + buf]);
        }
        mma_commit(&bar[EX_AEMPTY]);  // the latent rows may be replaced once these MMAs are done
      }
      mma_commit(&bar[EX_DRAIN]);
      mbar_wait_drain(&bar[EX_DRAIN], 0, wc);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- epilogue
    const int q4 = warp & 3, r = q4 * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    uint32_t e = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const ExUnit un = ex_unit(p, u);
      const int row = un.row0 + r;
      for (int j = un.j0; j < un.j1; ++j, ++e) {
        const uint32_t buf = e % 4;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar[EX_DFULL + buf], (e / 4) & 1u, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int h = j < p.H ? j : j - p.H;
        uint4* dst = reinterpret_cast<uint4*>((j < p.H ? p.k_c : p.v_c) + ((size_t)row * p.H + h) * 128);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tl + buf * 128 + (uint32_t)(c * 32), v);
          tmem_wait_ld();
          if (row < p.T) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[c * 4 + q] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                  pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                  pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                  pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          }
        }
        tc_fence_before();
        mbar_arrive(&bar[EX_DEMPTY + buf]);
      }
    }
  }

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
