// append.cuh -- the cache-append step: each new token's latent c and rotated
// RoPE key, written into the latent cache at the token's position.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / KeyValue":
//   c_t^KV = W^DKV h_t   (W^DKV in R^{d_c x d}),
//   k_t^R  = RoPE_t(W^KR h_t)   (W^KR in R^{d_h^R x d}),
// and (c_t^KV, k_t^R) is all a token leaves in the cache.
//
// The down-projection is [B*S x d] x [d x 576].  Few tokens, a long d: the
// weight takes the MMA's M slot (four 128-row tiles of W^DKV and one tile of
// the 64 rows of W^KR), the tokens take N, and d is cut into slices of
// kAppKc columns, one CTA per (weight tile, slice, token tile), so that about
// a hundred SMs stream the 8 MB of weights at once.  Each CTA leaves its fp32
// partial product in a workspace; the finalize sums the slices in a fixed
// order (the result does not depend on timing), rotates the k^R part at the
// token's position (fp64 angle reduction, as rope.cuh) and writes both parts,
// rounded to bf16, into the cache rows.  When all CTAs fit on the GPU at once
// the finalize runs in the same (cooperative) launch after a grid-wide
// barrier; otherwise a second kernel does it.
#pragma once

#include "rope.cuh"
#include "sm100.cuh"

namespace mla {

constexpr int kAppThreads = 128;
constexpr int kAppKc = 256;    // d columns per CTA: four 64-column atoms
constexpr int kAppCols = 576;  // d_c + d_h^R

struct AppendFinalizeParams {
  const float* part;       // [ks][BS][576]
  const int32_t* seqlens;  // [B]: the new tokens sit at seqlens[b] - S .. seqlens[b] - 1
  __nv_bfloat16* c_kv;     // [B, Lmax, 512]
  __nv_bfloat16* k_r;      // [B, Lmax, 64]
  uint32_t* status;
  int BS, S, ks, Lmax;
};

struct AppendParams {
  float* part;        // [ks][BS][576] fp32 partial products
  int BS, n_tile, ks;
  uint32_t tmem_cols;
  uint32_t* status;
  uint64_t timeout_ns;
  uint32_t* barrier;  // fused form: [0] arrivals, [1] generation (zero-filled workspace words)
  int fused;          // 1: finalize in this launch after a grid-wide barrier (cooperative launch)
  AppendFinalizeParams fin;
};

// Output pair t (0..287) of token n: the slices summed in order; pairs 0..255
// are c^KV, pairs 256..287 the k^R pairs, turned by pos * theta_j.
__device__ __forceinline__ void append_finalize_pair(const AppendFinalizeParams& p, const RopeTheta& th, int n,
                                                     int t) {
  const int b = n / p.S, s = n - b * p.S;
  const int64_t pos = (int64_t)p.seqlens[b] - p.S + s;
  if (pos < 0 || pos >= p.Lmax) {
    if (t == 0) atomicOr(p.status, kDevErrBadSeqlen);
    return;
  }
  const float2* src = reinterpret_cast<const float2*>(p.part + (size_t)n * kAppCols) + t;
  const size_t kstep = (size_t)p.BS * kAppCols / 2;  // float2 elements between slices
  // the slices (28 at d = 7168) are requested together, then summed in order;
  // read through L2 (.cg), since in the fused form they were written by this launch
  float x = 0.f, y = 0.f;
  for (int k0 = 0; k0 < p.ks; k0 += 32) {
    float2 v[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) v[u] = k0 + u < p.ks ? __ldcg(src + (size_t)(k0 + u) * kstep) : make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      x += v[u].x;
      y += v[u].y;
    }
  }
  if (t < 256) {
    reinterpret_cast<__nv_bfloat162*>(p.c_kv + ((size_t)b * p.Lmax + pos) * 512)[t] = __floats2bfloat162_rn(x, y);
  } else {
    const int j = t - 256;
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    const double a = (double)pos * th.theta[j];
    const double rr = fma(-rint(a * inv_two_pi), two_pi, a);
    float sn, cs;
    sincosf((float)rr, &sn, &cs);
    reinterpret_cast<__nv_bfloat162*>(p.k_r + ((size_t)b * p.Lmax + pos) * 64)[j] =
        __floats2bfloat162_rn(x * cs - y * sn, x * sn + y * cs);
  }
}

__host__ __device__ constexpr size_t app_smem_bytes(int n_tile) {
  return (size_t)4 * 16384 + (size_t)4 * n_tile * 128 + 64;
}

__global__ void __launch_bounds__(kAppThreads, 1)
    append_gemm_kernel(const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_wr,
                       const __grid_constant__ CUtensorMap tm_h, const AppendParams p, const RopeTheta th) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int mt = blockIdx.x;       // 0..3: W^DKV rows 128 mt ..; 4: W^KR
  const int split = blockIdx.y;    // d columns split * kAppKc ..
  const int n0 = blockIdx.z * p.n_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* sA = smem;
  uint8_t* sB = smem + 4 * 16384;
  const uint32_t bbytes = (uint32_t)p.n_tile * 128u;  // one atom of B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 4 * bbytes);  // [0] A, [1] B, [2] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init_cluster();
    tma_prefetch_desc(mt < 4 ? &tm_wd : &tm_wr);
    tma_prefetch_desc(&tm_h);
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
    // The weights are inputs of the step: they stream in before the wait.
    // W^KR has 64 rows; its 128-row box is filled with zeros past them.
    mbar_arrive_expect_tx(&bars[0], 4 * 16384);
    tma_load_3d(sA, mt < 4 ? &tm_wd : &tm_wr, &bars[0], 0, mt < 4 ? mt * 128 : 0, split * 4);
  }
  pdl_wait();  // h may come from the kernel before this one; part is read by the last finalize
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[1], 4 * bbytes);
    tma_load_3d(sB, &tm_h, &bars[1], 0, n0, split * 4);
    const bool ok = mbar_wait(&bars[0], 0, wc) && mbar_wait(&bars[1], 0, wc);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, 0, 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
      for (int k = 0; k < 16; ++k) {  // four atoms x four K-steps of 16
        const uint64_t ad = smem_desc(a0 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(b0 + (k >> 2) * bbytes + (k & 3) * 32, 16, 1024, 2);
        mma_ss(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(&bars[2]);
    }
  }
  __syncwarp();
  const bool ok = mbar_wait(&bars[2], 0, wc);
  tc_fence_after();
  if (ok) {
    const int m = warp * 32 + lane;  // weight row in the tile = output column
    const int col = mt < 4 ? mt * 128 + m : 512 + m;
    const bool live = mt < 4 || m < 64;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const int nvalid = min(p.n_tile, p.BS - n0);
    float* dst = p.part + ((size_t)split * p.BS + n0) * kAppCols + col;
    for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tl + (uint32_t)c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (live && c0 + c < nvalid) dst[(size_t)(c0 + c) * kAppCols] = __uint_as_float(r[c]);
    }
  }
  __threadfence();  // the partial product is visible device-wide before this CTA arrives below
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (!p.fused) return;
  // Fused form (a cooperative launch: every CTA is resident): a grid-wide
  // barrier on two workspace words -- arrivals, reset by the last CTA to
  // arrive, which then bumps the generation the others wait on (bounded) --
  // and then every CTA finalizes its share of the output pairs.
  volatile uint32_t* go = tmem_slot;  // reused: 1 = the barrier completed
  if (threadIdx.x == 0) {
    const uint32_t total = gridDim.x * gridDim.y * gridDim.z;
    volatile uint32_t* gen = p.barrier + 1;
    const uint32_t g0 = *gen;
    uint32_t passed = 1u;
    if (atomicAdd(p.barrier, 1u) == total - 1u) {
      atomicExch(p.barrier, 0u);
      __threadfence();
      atomicAdd(p.barrier + 1, 1u);
    } else {
      const uint64_t t0 = global_timer_ns();
      while (*gen == g0) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          atomicOr(p.status, kDevErrTimeout);
          passed = 0u;
          break;
        }
        __nanosleep(100);
      }
    }
    __threadfence();
    *go = passed;
  }
  __syncthreads();
  if (!*go) return;
  const int total = (int)(gridDim.x * gridDim.y * gridDim.z);
  const int cta = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int pairs = p.BS * (kAppCols / 2);
  for (int i = cta * kAppThreads + (int)threadIdx.x; i < pairs; i += total * kAppThreads)
    append_finalize_pair(p.fin, th, i / (kAppCols / 2), i % (kAppCols / 2));
}

// Block = one token, thread = one pair of output columns (288 per token).
__global__ void __launch_bounds__(kAppCols / 2)
    append_finalize_kernel(const AppendFinalizeParams p, const RopeTheta th) {
  pdl_trigger();
  pdl_wait();  // the partial products come from the GEMM kernel
  append_finalize_pair(p, th, blockIdx.x, threadIdx.x);
}

}  // namespace mla
