// combine_up.cuh -- the split-KV merge fused into the up-projection.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention":
//   o_lat = sum_j a_j c_j with ONE softmax over all visible positions
//   ("注意力计算"), then o = W^UV_h o_lat ("潜在向量的作用").
// The decode kernel leaves each sequence's o_lat as split-KV partials
// (splitkv.cuh): per segment k and query row, its reference exponent m_k,
// its sum l_k and the normalised mix U_k (fp16).  This kernel merges them,
//   o_lat = sum_k w_k U_k / sum_k w_k,   w_k = l_k 2^(m_k - M),
// straight into the shared-memory operand of the up-projection MMA, so o_lat
// never goes to memory.  (Measured inside the pipelined step on B300 it is
// slower than the two kernels it replaces, about 87.5 against 83.5 us per
// step at B = 32, L = 4096: its 1024-thread CTAs start only on SMs the decode
// has left entirely, while the small combine CTAs sit ready beside the
// decode.  The step therefore keeps the two launches; this entry serves
// callers that hold no o_lat buffer.)
//
// One CTA owns one head h and a tile of n_tile <= 32 query rows, one warp
// per row.  W^UV_h (128 KB) streams in by TMA before the dependency wait,
// while the decode kernel finishes.  After it, each warp requests its row's
// (m, l) of every segment (lanes over segments) together with the first two
// segments' partial rows (lanes over column octets), so a row with up to two
// segments costs one memory round trip; the rest follow two segments at a
// time.  The merged row is rounded to bf16 and written in the 128-byte
// swizzled K-major layout the MMA reads; then the MMA and epilogue follow
// up_project.cuh.
#pragma once

#include "splitkv.cuh"

namespace mla {

constexpr int kCUTile = 32;    // query rows per CTA (one warp each)
constexpr int kCUSegLanes = 3;  // segments per row handled: 32 * 3 = 96 >= G

struct CombineUpParams {
  const int32_t* prefix;  // plan (splitkv.cuh)
  const int32_t* gfirst;
  const int32_t* segbase;
  const float2* ml;       // [slots * n_rb, 128]
  const uint4* opart;     // [slots * n_rb][64 column octets][128 rows] fp16 x 8 (2^-e U)
  const uint8_t* oexp;    // [slots * n_rb][128 rows][2 halves] e
  const uint32_t* plan_ok;
  __nv_bfloat16* out;     // [BS, H, 128]
  int B, S, H, n_rb, G, BS, n_tile;  // n_tile: multiple of 16, <= kCUTile
  uint32_t tmem_cols;
  uint32_t* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t cu_smem_bytes(int n_tile) {
  return (size_t)8 * 16384 + (size_t)8 * n_tile * 128 + 128;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void acc_f16x8(float (&acc)[8], const uint4& x, float w) {
  const uint32_t* h = reinterpret_cast<const uint32_t*>(&x);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
    acc[2 * e] += w * f.x;
    acc[2 * e + 1] += w * f.y;
  }
}

__global__ void __launch_bounds__(kCUTile * 32, 1)
    combine_up_kernel(const __grid_constant__ CUtensorMap tm_w, const CombineUpParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int h = blockIdx.x;
  const int n0 = blockIdx.y * p.n_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* sA = smem;
  uint8_t* sB = smem + 8 * 16384;
  const uint32_t bbytes = (uint32_t)p.n_tile * 128u;  // one atom of B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 8 * bbytes);  // [0..3] weight boxes, [4] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init_cluster();
    tma_prefetch_desc(&tm_w);
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
    // this one: it streams in while that kernel finishes.
    for (int a = 0; a < 4; ++a) {
      mbar_arrive_expect_tx(&bars[a], 32768u);
      tma_load_3d(sA + a * 32768, &tm_w, &bars[a], 0, h * 128, a * 2);
    }
  }
  pdl_wait();  // the partials and the plan come from the decode kernel

  // ---------------------------------------------------- merge: warp = row n
  if (warp < p.n_tile) {
    const int n = warp, q = n0 + n;
    float acc[2][8];
#pragma unroll
    for (int o = 0; o < 2; ++o)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[o][e] = 0.f;
    float inv = 0.f;
    if (q < p.BS && *p.plan_ok != 0u) {
      const int b = q / p.S, s = q - b * p.S;
      const int gr = s * p.H + h, rb = gr >> 7, r = gr & 127;
      const int k0 = p.segbase[b], ns = p.segbase[b + 1] - k0, g0 = p.gfirst[b];
      const int64_t T = p.prefix[p.B];
      const bool may_be_empty = T < p.G;  // only then can a group own no tile
      const uint4* urow = p.opart + (size_t)rb * 64 * 128 + r;  // + (k n_rb 64 + octet) 128
      const size_t kstride = (size_t)p.n_rb * 64 * 128;
      // (m, l) of segments lane + 32 u, and the first two segments' columns,
      // requested together
      float2 v[kCUSegLanes];
#pragma unroll
      for (int u = 0; u < kCUSegLanes; ++u) {
        const int j = lane + 32 * u;
        v[u] = (j < ns && !(may_be_empty && group_empty(g0 + j, T, p.G)))
                   ? __ldg(&p.ml[((size_t)(k0 + j) * p.n_rb + rb) * 128 + r])
                   : make_float2(0.f, 0.f);
      }
      uint4 x[2][2];
      uint32_t ex2[2];  // the two half-row exponents of a segment (octets 0..31, 32..63)
      const uint16_t* erow = reinterpret_cast<const uint16_t*>(p.oexp) + (size_t)rb * 128 + r;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int o = 0; o < 2; ++o)
          x[j][o] = j < ns ? __ldg(urow + (size_t)(k0 + j) * kstride + (size_t)(lane + 32 * o) * 128)
                           : make_uint4(0u, 0u, 0u, 0u);
        ex2[j] = j < ns ? (uint32_t)__ldg(erow + (size_t)(k0 + j) * p.n_rb * 128) : 0u;
      }
      float M = -INFINITY;
#pragma unroll
      for (int u = 0; u < kCUSegLanes; ++u)
        if (v[u].y > 0.f) M = fmaxf(M, v[u].x);
      M = warp_max(M);
      float w[kCUSegLanes], den = 0.f;
#pragma unroll
      for (int u = 0; u < kCUSegLanes; ++u) {
        w[u] = v[u].y > 0.f ? exp2f(v[u].x - M) * v[u].y : 0.f;  // the m are integers
        den += w[u];
      }
      den = warp_sum(den);
      inv = den > 0.f ? 1.f / den : 0.f;
      // weight of segment j, held by lane j % 32 in w[j / 32]
      auto weight = [&](int j) {
        const float a = __shfl_sync(0xffffffffu, w[0], j & 31);
        const float c = __shfl_sync(0xffffffffu, w[1], j & 31);
        const float d = __shfl_sync(0xffffffffu, w[2], j & 31);
        return j < 32 ? a : (j < 64 ? c : d);
      };
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float wj = weight(j);
        if (j < ns && wj != 0.f)  // empty groups' slots hold arbitrary bytes
#pragma unroll
          for (int o = 0; o < 2; ++o) acc_f16x8(acc[o], x[j][o], wj * pow2i((int)((ex2[j] >> (8 * o)) & 0xFFu)));
      }
      for (int j = 2; j < ns; j += 2) {  // further segments, two at a time
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
          for (int o = 0; o < 2; ++o)
            x[jj][o] = j + jj < ns ? __ldg(urow + (size_t)(k0 + j + jj) * kstride + (size_t)(lane + 32 * o) * 128)
                                   : make_uint4(0u, 0u, 0u, 0u);
          ex2[jj] = j + jj < ns ? (uint32_t)__ldg(erow + (size_t)(k0 + j + jj) * p.n_rb * 128) : 0u;
        }
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float wj = weight(j + jj);
          if (j + jj < ns && wj != 0.f)
#pragma unroll
            for (int o = 0; o < 2; ++o)
              acc_f16x8(acc[o], x[jj][o], wj * pow2i((int)((ex2[jj] >> (8 * o)) & 0xFFu)));
        }
      }
    }
    // octet lane + 32 o of row n: atom (octet / 8), 16-byte chunk (octet % 8) ^ (n % 8)
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int oct = lane + 32 * o;
      *reinterpret_cast<uint4*>(sB + (oct >> 3) * bbytes + n * 128 + (((oct & 7) ^ (n & 7)) << 4)) =
          make_uint4(pack_bf16x2(acc[o][0] * inv, acc[o][1] * inv), pack_bf16x2(acc[o][2] * inv, acc[o][3] * inv),
                     pack_bf16x2(acc[o][4] * inv, acc[o][5] * inv), pack_bf16x2(acc[o][6] * inv, acc[o][7] * inv));
    }
  }
  fence_proxy_async_cta();  // the MMA reads the operand through the async proxy
  __syncthreads();

  // ---------------------------------------------------- up-projection
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    bool ok = true;
    for (int a = 0; a < 4 && ok; ++a) {
      ok = mbar_wait(&bars[a], 0, wc);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // two atoms x four K-steps of 16
        const int atom = a * 2 + (k >> 2);
        const uint64_t ad = smem_desc(a0 + atom * 16384 + (k & 3) * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(b0 + atom * bbytes + (k & 3) * 32, 16, 1024, 2);
        mma_ss(tmem, ad, bd, idesc, (a | k) ? 1u : 0u);
      }
    }
    if (ok) mma_commit(&bars[4]);
  }
  if (warp < 4) {
    __syncwarp();
    const bool ok = mbar_wait(&bars[4], 0, wc);
    tc_fence_after();
    if (ok) {
      const int v = warp * 32 + lane;
      const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
      const int nvalid = min(p.n_tile, p.BS - n0);
      for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
        uint32_t rr[16];
        tmem_ld16(tl + c0, rr);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c0 + c < nvalid)
            p.out[((size_t)(n0 + c0 + c) * p.H + h) * 128 + v] = __float2bfloat16_rn(__uint_as_float(rr[c]));
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
