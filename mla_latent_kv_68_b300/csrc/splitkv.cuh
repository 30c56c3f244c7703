// splitkv.cuh -- split-KV plan and log-sum-exp combine.
//
// The softmax of "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent
// Attention / 注意力计算" normalises once over all visible positions.  The
// decode kernel cuts every sequence's cache rows into contiguous runs of
// 128-row tiles ("segments") spread over all SMs; each segment k leaves, per
// query row, its reference exponent m_k (an integer, log2 units), the sum
// l_k = sum_j 2^(s2_j - m_k) and the normalised latent mix
// U_k = sum_j 2^(s2_j - m_k) c_j / l_k, stored in fp16 as 2^-e U_k with one
// exponent e >= 0 per row and 256-column half that keeps it in fp16 range.
// Merging them restores the single normalisation:
//     o_lat = sum_k w_k U_k / sum_k w_k,   w_k = 2^(m_k - M) l_k,   M = max_k m_k.
//
// Tiles are kTileRows = 128 cache rows (the N of the decode's QK^T MMAs).
// Plan: the cache tiles of all sequences are laid end to end (sequence-major),
// each sequence's tiles after one unit that stands for the cost of starting
// it, and the T units are cut into G equal runs, one per group of clusters.
// Group g owns units [floor(g T / G), floor((g+1) T / G)).  A sequence b
// contributes one segment to every group its tiles touch; its segments get
// consecutive slot numbers starting at segbase[b].  The decode kernel works the plan out
// itself from the sequence lengths (decode.cuh, plan_scan) and leaves the
// arrays below (prefix, gfirst, segbase, plan_ok) for the combine.
#pragma once

#include "sm100.cuh"

namespace mla {

constexpr int kTileRows = 128;

__device__ __forceinline__ int tiles_of(int L) { return (L + kTileRows - 1) / kTileRows; }

// Group owning flat tile x: the largest g with floor(g T / G) <= x.
__device__ __forceinline__ int group_of(int64_t x, int64_t T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

struct CombineParams {
  const int32_t* prefix;   // plan: prefix[b] = the unit of b's first tile, prefix[B] = total units T
  const int32_t* gfirst;
  const int32_t* segbase;
  const float2* ml;     // [slots * n_rb, 128] (m_k, l_k)
  const uint4* opart;   // [slots * n_rb][64 column octets][128 rows] fp16 x 8 (2^-e U_k)
  const uint8_t* oexp;  // [slots * n_rb][128 rows][2 halves] e
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
// loads of a thread do not depend on one another: the (m, l) and the columns
// of up to kSegBatch segments are requested together, so a row block with
// that many segments costs one memory round trip, and longer ones fold batch
// after batch into running sums kept relative to the largest m so far.
constexpr int kCombineCols = 32;
constexpr int kSegBatch = 4;

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
  const bool may_be_empty = T < p.G;  // only then can a group own no tile

  float M = -INFINITY, den = 0.f;
  float acc[kCombineCols];
#pragma unroll
  for (int i = 0; i < kCombineCols; ++i) acc[i] = 0.f;
  const int half = c0 >> 8;  // which exponent of the row applies to these columns
  for (int kb = k0; kb < k1; kb += kSegBatch) {
    float2 ml[kSegBatch];
    int ee[kSegBatch];
    uint4 x[kSegBatch][kCombineCols / 8];
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      const int k = kb + u;
      const bool ok = k < k1 && !(may_be_empty && group_empty(g0 + k - k0, T, p.G));
      const size_t idx = (size_t)k * p.n_rb + rb;
      ml[u] = ok ? __ldg(&p.ml[idx * 128 + r]) : make_float2(0.f, 0.f);
      ee[u] = ok ? (int)__ldg(&p.oexp[(idx * 128 + r) * 2 + half]) : 0;
#pragma unroll
      for (int c = 0; c < kCombineCols / 8; ++c)
        x[u][c] = ok ? __ldg(p.opart + (idx * 64 + c0 / 8 + c) * 128 + r) : make_uint4(0u, 0u, 0u, 0u);
    }
    float Mb = M;
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u)
      if (ml[u].y > 0.f) Mb = fmaxf(Mb, ml[u].x);
    if (Mb > M) {  // the m are integers: exact powers of two
      const float sc = M == -INFINITY ? 0.f : exp2f(M - Mb);
      den *= sc;
#pragma unroll
      for (int i = 0; i < kCombineCols; ++i) acc[i] *= sc;
      M = Mb;
    }
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      if (!(ml[u].y > 0.f)) continue;  // no segment, or no visible row in it
      const float w = exp2f(ml[u].x - M) * ml[u].y;
      den += w;
      const float wu = w * pow2i(ee[u]);  // the stored partial is 2^-e U
#pragma unroll
      for (int c = 0; c < kCombineCols / 8; ++c) {
        const uint32_t* h = reinterpret_cast<const uint32_t*>(&x[u][c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
          acc[8 * c + 2 * e] += wu * f.x;
          acc[8 * c + 2 * e + 1] += wu * f.y;
        }
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
