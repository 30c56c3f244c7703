// splitkv.cuh -- split-KV plan and log-sum-exp combine.
//
// The softmax of "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent
// Attention / 注意力计算" normalises once over all visible positions.  The
// decode kernel cuts every sequence's cache rows into contiguous runs of
// 128-row tiles ("segments") spread over all SMs; each segment k leaves, per
// query row, its reference exponent m_k (an integer, log2 units), the sum
// l_k = sum_j 2^(s2_j - m_k) and the normalised latent mix
// U_k = sum_j 2^(s2_j - m_k) c_j / l_k (fp16).  Merging them restores the
// single normalisation:
//     o_lat = sum_k w_k U_k / sum_k w_k,   w_k = 2^(m_k - M) l_k,   M = max_k m_k.
//
// Tiles are kTileRows = 128 cache rows (the N of the decode's QK^T MMAs).
// Plan: the cache tiles of all sequences are laid end to end (sequence-major)
// and cut into G equal runs, one per group of clusters.  Group g owns flat
// tiles [floor(g T / G), floor((g+1) T / G)).  A sequence b contributes one
// segment to every group its tiles touch; its segments get consecutive slot
// numbers starting at segbase[b].
#pragma once

#include "sm100.cuh"

namespace mla {

struct PlanParams {
  const int32_t* seqlens;
  int B, S, Lmax, G;
  int32_t* prefix;   // [B+1] exclusive prefix of tiles per sequence; prefix[B] = T
  int32_t* gfirst;   // [B] first group touching sequence b
  int32_t* segbase;  // [B+1] exclusive prefix of segments per sequence
  int32_t* gstart;   // [G] first sequence touched by each group
  uint32_t* status;
  uint32_t* plan_ok;
};

constexpr int kTileRows = 128;

__device__ __forceinline__ int tiles_of(int L) { return (L + kTileRows - 1) / kTileRows; }

// Group owning flat tile x: the largest g with floor(g T / G) <= x.
__device__ __forceinline__ int group_of(int64_t x, int64_t T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += t;
    }
    if (lane < nw) warp_sums[lane] = winc - w;
    if (lane == nw - 1) warp_sums[32] = winc;
  }
  __syncthreads();
  const int excl = warp_sums[warp] + inc - v;
  *total = warp_sums[32];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(1024) plan_kernel(const PlanParams p) {
  __shared__ int warp_sums[33];
  __shared__ int bad;
  pdl_trigger();
  pdl_wait();  // the workspace may still be read by the previous step's kernels
  const int nt = blockDim.x;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  const int E = (p.B + nt - 1) / nt;
  const int beg = min(p.B, (int)threadIdx.x * E), end = min(p.B, beg + E);

  int local = 0;
  for (int b = beg; b < end; ++b) {
    const int L = p.seqlens[b];
    if (L < p.S || L > p.Lmax) bad = 1;
    else local += tiles_of(L);
  }
  int T;
  int run = block_exclusive_scan(local, warp_sums, &T);
  for (int b = beg; b < end; ++b) {
    p.prefix[b] = run;
    const int L = p.seqlens[b];
    if (L >= p.S && L <= p.Lmax) run += tiles_of(L);
  }
  if (threadIdx.x == 0) p.prefix[p.B] = T;
  __syncthreads();

  local = 0;
  for (int b = beg; b < end; ++b) {
    const int x0 = p.prefix[b], x1 = p.prefix[b + 1];
    int ns = 0, gf = 0;
    if (x1 > x0) {
      gf = group_of(x0, T, p.G);
      ns = group_of(x1 - 1, T, p.G) - gf + 1;
    }
    p.gfirst[b] = gf;
    local += ns;
  }
  int nseg_total;
  run = block_exclusive_scan(local, warp_sums, &nseg_total);
  for (int b = beg; b < end; ++b) {
    p.segbase[b] = run;
    const int x0 = p.prefix[b], x1 = p.prefix[b + 1];
    if (x1 > x0) run += group_of(x1 - 1, T, p.G) - group_of(x0, T, p.G) + 1;
  }
  for (int g = threadIdx.x; g < p.G; g += nt) {  // largest b with prefix[b] <= floor(g T / G)
    const int64_t tg = (int64_t)g * T / p.G;
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.prefix[mid] <= tg) lo = mid;
      else hi = mid - 1;
    }
    p.gstart[g] = lo;
  }
  if (threadIdx.x == 0) {
    p.segbase[p.B] = nseg_total;
    *p.plan_ok = bad ? 0u : 1u;
    if (bad) atomicOr(p.status, kDevErrBadSeqlen);
  }
}

struct CombineParams {
  const int32_t* prefix;   // plan: prefix[B] = total tiles T
  const int32_t* gfirst;
  const int32_t* segbase;
  const float2* ml;     // [slots * n_rb, 128] (m_k, l_k)
  const uint4* opart;   // [slots * n_rb][64 column octets][128 rows] fp16 x 8 (U_k)
  __nv_bfloat16* o_lat; // [B*S*H, 512]
  const uint32_t* plan_ok;
  int B, S, H, n_rb, G;
};

// Group g of G owns flat tiles [floor(g T / G), floor((g+1) T / G)); when
// T < G some groups own none.  A sequence's segment slots cover every group
// from its first to its last, so a slot of an empty group is never written
// by the decode and must be skipped.
__device__ __forceinline__ bool group_empty(int g, int64_t T, int G) {
  return (int64_t)g * T / G == (int64_t)(g + 1) * T / G;
}

// Block = one 128-row block of one sequence and kCombineCols latent columns;
// thread = one query row.  Partials are stored as column octets x rows of
// 8 fp16, so every 16-byte load of a warp reads 512 consecutive bytes.  The
// (m, l) of all segments are read first; the partial columns of two segments
// are then loaded together so that the few L2 round trips of a row overlap.
constexpr int kCombineCols = 32;

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  pdl_trigger();
  pdl_wait();  // the partials come from the decode kernel
  const int b = blockIdx.x / p.n_rb, rb = blockIdx.x - b * p.n_rb;
  const int c0 = blockIdx.y * kCombineCols;
  const int r = threadIdx.x;
  const int SH = p.S * p.H;
  if (c0 >= 512 || rb * 128 + r >= SH) return;
  if (*p.plan_ok == 0u) return;
  const int k0 = p.segbase[b], k1 = p.segbase[b + 1], g0 = p.gfirst[b];
  const int64_t T = p.prefix[p.B];

  float M = -INFINITY;
  for (int k = k0; k < k1; ++k) {
    if (group_empty(g0 + k - k0, T, p.G)) continue;
    const float2 v = p.ml[((size_t)k * p.n_rb + rb) * 128 + r];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float acc[kCombineCols];
#pragma unroll
  for (int i = 0; i < kCombineCols; ++i) acc[i] = 0.f;
  float den = 0.f;
  for (int k = k0; k < k1; k += 2) {
    float w[2];
    const uint4* src[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kk = k + u;
      w[u] = 0.f;
      src[u] = p.opart;
      if (kk < k1 && !group_empty(g0 + kk - k0, T, p.G)) {
        const size_t idx = (size_t)kk * p.n_rb + rb;
        const float2 v = p.ml[idx * 128 + r];
        if (v.y > 0.f) {
          w[u] = exp2f(v.x - M) * v.y;
          den += w[u];
          src[u] = p.opart + (idx * 64 + c0 / 8) * 128 + r;
        }
      }
    }
    uint4 x[2][kCombineCols / 8];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int c = 0; c < kCombineCols / 8; ++c)
        x[u][c] = w[u] != 0.f ? __ldg(src[u] + (size_t)c * 128) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < kCombineCols / 8; ++c) {
      const uint32_t* a = reinterpret_cast<const uint32_t*>(&x[0][c]);
      const uint32_t* b = reinterpret_cast<const uint32_t*>(&x[1][c]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a[e]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b[e]));
        acc[8 * c + 2 * e] += w[0] * fa.x + w[1] * fb.x;
        acc[8 * c + 2 * e + 1] += w[0] * fa.y + w[1] * fb.y;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(p.o_lat + ((size_t)b * SH + rb * 128 + r) * 512 + c0);
#pragma unroll
  for (int q = 0; q < kCombineCols / 8; ++q)
    dst[q] = make_uint4(pack_bf16x2(acc[8 * q] * inv, acc[8 * q + 1] * inv),
                        pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                        pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                        pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
}

}  // namespace mla
