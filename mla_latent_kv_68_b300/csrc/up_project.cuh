// up_project.cuh -- o = W^UV_h o_lat per head, on the tcgen05 tensor cores.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention /
// 潜在向量的作用": o_{t,i} = W_i^UV (sum_j a_{t,j,i} c_j), i.e. values are
// aggregated in latent space and projected up once per query.
//
// Per head h this is [B*S x 512] x [512 x 128]; the weight again takes the
// MMA's M slot:  D[v, n] = sum_k W_UV[h][v][k] * o_lat[n][h][k]
// (M = v = 128, N = n, K = k = 512), both operands K-major.  One CTA owns one
// head and one tile of up to 64 query rows.  The weight (128 KB) arrives as
// four 32 KB TMA boxes of two 64-wide k atoms each, on their own barriers, so
// the MMAs start on the first one; the query rows' eight k atoms come in one
// 4-D box.  Large boxes matter on B300: an SM's TMA unit sustains a few boxes
// per microsecond.
//
// Shared memory (128-byte swizzle): A 8 x [128 v][64 k] = 128 KB,
// B 8 x [n_tile][64 k] = n_tile KB.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kUpThreads = 128;

struct UpParams {
  __nv_bfloat16* out;  // [BS, H, 128]
  int BS, H, n_tile;   // n_tile: multiple of 16, <= 64
  uint32_t tmem_cols;  // power of two >= max(32, n_tile)
  uint32_t* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t up_smem_bytes(int n_tile) {
  return (size_t)8 * 16384 + (size_t)8 * n_tile * 128 + 128;
}

__global__ void __launch_bounds__(kUpThreads, 1)
    up_project_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_o, const UpParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int h = blockIdx.x;
  const int n0 = blockIdx.y * p.n_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* sA = smem;
  uint8_t* sB = smem + 8 * 16384;
  const uint32_t bbytes = (uint32_t)p.n_tile * 128u;  // one atom of B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 8 * bbytes);  // [0..3] weight boxes, [4] o, [5] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_trigger();
  if (threadIdx.x == 0) {
    // The weight is an input of the step, not an output of the kernel before
    // this one: it streams in while that kernel finishes.  o_lat is.
    for (int a = 0; a < 4; ++a) {
      mbar_arrive_expect_tx(&bars[a], 32768u);
      tma_load_3d(sA + a * 32768, &tm_w, &bars[a], 0, h * 128, a * 2);
    }
    pdl_wait();
    mbar_arrive_expect_tx(&bars[4], 8 * bbytes);
    tma_load_4d(sB, &tm_o, &bars[4], 0, n0, 0, h);
    const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    bool ok = mbar_wait(&bars[4], 0, wc);
    for (int a = 0; a < 4 && ok; ++a) {
      ok = mbar_wait(&bars[a], 0, wc);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int w = 0; w < 8; ++w) {  // two atoms x four K-steps of 16
        const int atom = a * 2 + (w >> 2);
        const uint64_t ad = smem_desc(a0 + atom * 16384 + (w & 3) * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(b0 + atom * bbytes + (w & 3) * 32, 16, 1024, 2);
        mma_ss(tmem, ad, bd, idesc, (a | w) ? 1u : 0u);
      }
    }
    if (ok) mma_commit(&bars[5]);
  }
  __syncwarp();
  pdl_wait();  // every thread, before its first global write

  const bool ok = mbar_wait(&bars[5], 0, wc);
  tc_fence_after();
  if (ok) {
    const int v = warp * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const int nvalid = min(p.n_tile, p.BS - n0);
    for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tl + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c0 + c < nvalid)
          p.out[((size_t)(n0 + c0 + c) * p.H + h) * 128 + v] =
              __float2bfloat16_rn(__uint_as_float(r[c]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

}  // namespace mla
