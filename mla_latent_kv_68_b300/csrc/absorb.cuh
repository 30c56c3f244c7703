// absorb.cuh -- q~ = (W^UK_h)^T q^C per head on the tcgen05 tensor cores,
// optionally fused with the query RoPE.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention /
// 潜在向量的作用": (q^C)^T W^UK c = ((W^UK)^T q^C)^T c, so the key
// up-projection moves onto the query once per decode step.  The query's
// RoPE half ("Query": q^R = RoPE(W^QR c^Q) at the query position) is the other
// part of q_cat and is rotated here too when asked for, so one launch fills
// the whole q_cat row.
//
// Per head h this is [B*S x 128] x [128 x 512].  B*S is small (1..256 per
// tile), so the weight goes in the MMA's M slot: the kernel computes
//     D[k, n] = sum_d W_UK[h][d][k] * q_nope[n][h][d]      (M = k, N = n, K = d)
// with A = W_UK[h] read as an MN-major operand (k is contiguous in memory)
// and B = the q^C rows as a K-major operand.  One CTA owns one head, one half
// (256) of k as two M = 128 tiles, and one tile of up to 256 query rows; fp32
// accumulates in tensor memory and the epilogue rounds to bf16 into
// q_cat[n][h][k].  The weight half (64 KB) arrives as two 32 KB TMA boxes:
// on B300 an SM's TMA unit sustains a few boxes per microsecond, so the box
// size sets the bandwidth a weight-streaming kernel can reach.
//
// Shared memory (128-byte swizzle, 1024-byte aligned):
//   A: 4 atoms x [128 d][64 k] bf16            64 KB
//   B: 2 atoms x [n_tile rows][64 d] bf16      n_tile * 256 B
#pragma once

#include "rope.cuh"
#include "sm100.cuh"

namespace mla {

constexpr int kAbsorbThreads = 128;
constexpr int kAbsorbSmemA = 65536;

struct AbsorbParams {
  __nv_bfloat16* q_cat;            // [BS, H, 576]
  const __nv_bfloat16* q_rope;     // [BS, H, 64]; null: no RoPE (columns 512.. untouched)
  const int32_t* seqlens;          // [B] query positions seqlens[b] - S + s (RoPE only)
  int BS, S, H, n_tile;            // n_tile: multiple of 16, <= 256
  uint32_t tmem_cols;              // power of two >= max(32, 2 * n_tile)
  uint32_t* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t absorb_smem_bytes(int n_tile) {
  return (size_t)kAbsorbSmemA + (size_t)n_tile * 256 + 64;
}

__global__ void __launch_bounds__(kAbsorbThreads, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                  const AbsorbParams p, const RopeTheta th) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int h = blockIdx.x;
  const int half = blockIdx.y;             // k columns half * 256 .. + 255
  const int n0 = blockIdx.z * p.n_tile;    // first query row of this tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* sA = smem;
  uint8_t* sB = smem + kAbsorbSmemA;
  const uint32_t abytes = (uint32_t)p.n_tile * 128u;  // one 64-wide d atom of B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 2 * abytes);  // [0] full, [1] mma done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_q);
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
  pdl_wait();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], (uint32_t)kAbsorbSmemA + 2 * abytes);
    for (int a = 0; a < 2; ++a) {  // two 32 KB weight boxes: 2 atoms of 64 k each
      tma_load_3d(sA + a * 32768, &tm_w, &bars[0], 0, h * 128, half * 4 + a * 2);
      tma_load_3d(sB + a * abytes, &tm_q, &bars[0], a * 64, h, n0);
    }
  }

  // The query RoPE overlaps the weight load: the two k-halves' CTAs share it,
  // warps 1..3 do it (warp 0 issues the MMA as soon as the weight lands), and
  // each thread requests all its rows' positions and values before it
  // computes, so the loads cost one memory round trip rather than one each.
  const int nvalid = min(p.n_tile, p.BS - n0);
  if (p.q_rope != nullptr && warp >= 1) {
    constexpr int kRopeThreads = kAbsorbThreads - 32, kRopeBatch = 6;
    const int items = nvalid * 8, lo = half == 0 ? 0 : items / 2, hi = half == 0 ? items / 2 : items;
    for (int base = lo + (int)threadIdx.x - 32; base < hi; base += kRopeThreads * kRopeBatch) {
      int64_t pos[kRopeBatch];
      uint4 v[kRopeBatch];
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int it = base + u * kRopeThreads;
        pos[u] = -1;
        if (it < hi) {
          const int n = n0 + (it >> 3), b = n / p.S, s = n - b * p.S;
          pos[u] = (int64_t)p.seqlens[b] - p.S + s;
          v[u] = *reinterpret_cast<const uint4*>(p.q_rope + ((size_t)n * p.H + h) * 64 + (it & 7) * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int it = base + u * kRopeThreads;
        if (it < hi && pos[u] >= 0) {
          const int n = n0 + (it >> 3);
          *reinterpret_cast<uint4*>(p.q_cat + ((size_t)n * p.H + h) * 576 + 512 + (it & 7) * 8) =
              rope_rotate4(v[u], pos[u], it & 7, th);
        }
      }
    }
  }

  if (threadIdx.x == 0) {
    if (mbar_wait(&bars[0], 0, wc)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, /*a_mn=*/1, /*b_mn=*/0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // K = 128 in steps of 16
          // A, MN-major: 16 d-rows per step (2048 B); the two 64-wide k atoms of
          // tile t sit 16 KB apart, starting at t * 32 KB.
          const uint64_t ad = smem_desc(a0 + t * 32768 + kk * 2048, 16384, 1024, 2);
          // B, K-major: step kk lies in atom kk/4 at a 32-byte offset inside the 128-byte row.
          const uint64_t bd = smem_desc(b0 + (kk >> 2) * abytes + (kk & 3) * 32, 16, 1024, 2);
          mma_ss(tmem + (uint32_t)(t * p.n_tile), ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
      }
      mma_commit(&bars[1]);
    }
  }
  __syncwarp();

  const bool ok = mbar_wait(&bars[1], 0, wc);
  tc_fence_after();
  if (ok) {
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    for (int t = 0; t < 2; ++t) {
      const int k = half * 256 + t * 128 + warp * 32 + lane;  // this thread's tensor-memory lane
      for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tl + (uint32_t)(t * p.n_tile + c0), r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int n = n0 + c0 + c;
          if (c0 + c < nvalid)
            p.q_cat[((size_t)n * p.H + h) * 576 + k] = __float2bfloat16_rn(__uint_as_float(r[c]));
        }
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

}  // namespace mla
