// wgemm.cuh -- the output projection of the attention layer: u = W x per
// token, for a weight W that is read once per step (a decode batch of a few
// dozen tokens against a weight of hundreds of MB).
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention /
// 注意力计算": u_t = W^O [o_{t,1}; ...; o_{t,H}], the heads' outputs
// concatenated; "DeepSeek-V3 技术报告精读" (oopvo.github.io), "MLA": the
// value up-projection W^UV can be absorbed into W^O.  Both are this GEMM:
//   x = out  [BS][H * 128],  W = W^O                     [d][H * 128], or
//   x = o_lat [BS][H * 512], W = W^O blockdiag(W_h^UV)   [d][H * 512].
//
// [BS x K] x [K x M] with M = d: the weight takes the MMA's M slot (128 rows
// per tile), the tokens take N (n_tile <= 64), and K is cut into ks slices,
// one CTA per (weight tile, slice, token tile); ks is chosen so that the grid
// fills the SMs two CTAs deep, slices differing by at most one chunk.  A CTA
// streams its slice of the weight through a ring of 32 KB TMA boxes (128 rows
// x 128 columns, two 128-byte-swizzle atoms) next to the tokens' matching
// columns, and accumulates in tensor memory.  With ks > 1 each CTA leaves its fp32 partial
// product in a workspace and wgemm_reduce_kernel sums the slices in a fixed
// order (the result does not depend on timing); with ks = 1 the CTA writes u.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kWgThreads = 128;  // 4 warps: TMA (warp 0), MMA (warp 1), all four in the epilogue
constexpr int kWgKc = 128;       // K columns per ring stage
constexpr int kWgStages = 2;    // ~97 KB of shared memory: two CTAs per SM
constexpr int kWgMaxTile = 64;   // tokens per CTA

struct WGemmParams {
  float* part;            // [ks][BS][M] fp32 partial products (ks > 1)
  __nv_bfloat16* out;     // [BS][M] (ks == 1)
  int BS, M, n_tile, ks, total_chunks;  // K / kWgKc chunks, cut into ks near-equal slices
  uint32_t tmem_cols;
  uint32_t* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr int wg_stage_bytes(int n_tile) { return 2 * 16384 + 2 * n_tile * 128; }
__host__ __device__ constexpr size_t wg_smem_bytes(int n_tile) {
  return (size_t)kWgStages * wg_stage_bytes(n_tile) + 1024;
}

__global__ void __launch_bounds__(kWgThreads, 1)
    wgemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const WGemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int mt = blockIdx.x, split = blockIdx.y, n0 = blockIdx.z * p.n_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sbytes = wg_stage_bytes(p.n_tile);
  const uint32_t xbytes = (uint32_t)p.n_tile * 128u;  // one atom of the token rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWgStages * sbytes);  // full[kWgStages], empty[..], done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kWgStages + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < 2 * kWgStages + 1; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
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
  const int c0 = (int)((int64_t)split * p.total_chunks / p.ks);  // this CTA's K chunks: [c0, c0 + chunks)
  const int chunks = (int)((int64_t)(split + 1) * p.total_chunks / p.ks) - c0;

  if (warp == 0 && lane == 0) {
    // The weight is an input of the layer: its first stages stream in before
    // the wait for the kernel that produced x.
    int issued = 0;
    for (; issued < kWgStages && issued < chunks; ++issued) {
      uint8_t* st = smem + issued * sbytes;
      mbar_arrive_expect_tx(&bars[issued], (uint32_t)sbytes);
      tma_load_3d(st, &tm_w, &bars[issued], 0, mt * 128, (c0 + issued) * 2);
    }
    pdl_wait();
    for (int j = 0; j < issued; ++j)
      tma_load_3d(smem + j * sbytes + 32768, &tm_x, &bars[j], 0, n0, (c0 + j) * 2);
    for (int j = issued; j < chunks; ++j) {
      const int s = j % kWgStages;
      if (!mbar_wait(&bars[kWgStages + s], (uint32_t)((j / kWgStages) - 1) & 1u, wc)) break;
      uint8_t* st = smem + s * sbytes;
      mbar_arrive_expect_tx(&bars[s], (uint32_t)sbytes);
      tma_load_3d(st, &tm_w, &bars[s], 0, mt * 128, (c0 + j) * 2);
      tma_load_3d(st + 32768, &tm_x, &bars[s], 0, n0, (c0 + j) * 2);
    }
    // every issued copy lands before the CTA winds down
    for (int j = max(0, chunks - kWgStages); j < chunks; ++j)
      mbar_wait_drain(&bars[j % kWgStages], (uint32_t)(j / kWgStages) & 1u, wc);
  } else if (warp == 1 && lane == 0) {
    pdl_wait();
    const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, 0, 0);
    for (int j = 0; j < chunks; ++j) {
      const int s = j % kWgStages;
      if (!mbar_wait(&bars[s], (uint32_t)(j / kWgStages) & 1u, wc)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + s * sbytes), b0 = a0 + 32768;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // two atoms x four K-steps of 16
        const uint64_t ad = smem_desc(a0 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(b0 + (k >> 2) * xbytes + (k & 3) * 32, 16, 1024, 2);
        mma_ss(tmem, ad, bd, idesc, (j > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(&bars[kWgStages + s]);  // the stage is free once these MMAs have read it
    }
    mma_commit(&bars[2 * kWgStages]);
    mbar_wait_drain(&bars[2 * kWgStages], 0, wc);
  } else {
    pdl_wait();  // every global write comes after the kernel before this one
  }
  __syncwarp();
  const bool ok = mbar_wait(&bars[2 * kWgStages], 0, wc);
  tc_fence_after();
  if (ok) {
    const int m = mt * 128 + warp * 32 + lane;  // this thread's tensor-memory lane = weight row
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const int nvalid = min(p.n_tile, p.BS - n0);
    for (int cc = 0; cc < p.n_tile; cc += 16) {
      uint32_t r[16];
      tmem_ld16(tl + (uint32_t)cc, r);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (cc + c >= nvalid) continue;
        const size_t o = (size_t)(n0 + cc + c) * p.M + m;
        if (p.ks == 1)
          p.out[o] = __float2bfloat16_rn(__uint_as_float(r[c]));
        else
          p.part[(size_t)split * p.BS * p.M + o] = __uint_as_float(r[c]);
      }
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

// u[n][m] = sum over the slices, in order, of part[k][n][m]; four columns per thread.
__global__ void __launch_bounds__(256) wgemm_reduce_kernel(const float* part, __nv_bfloat16* out, int BS, int M,
                                                           int ks) {
  pdl_trigger();
  pdl_wait();  // the partial products come from wgemm_kernel
  const size_t total4 = (size_t)BS * M / 4;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total4) return;
  const float4* src = reinterpret_cast<const float4*>(part) + i;
  const size_t step = total4;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < ks; ++k) {
    const float4 v = __ldg(src + (size_t)k * step);
    a.x += v.x;
    a.y += v.y;
    a.z += v.z;
    a.w += v.w;
  }
  uint2 o;
  o.x = pack_bf16x2(a.x, a.y);
  o.y = pack_bf16x2(a.z, a.w);
  reinterpret_cast<uint2*>(out)[i] = o;
}

}  // namespace mla
