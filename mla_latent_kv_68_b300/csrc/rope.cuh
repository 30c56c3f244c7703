// rope.cuh -- rotary position embedding on interleaved pairs.
//
// "DeepSeek-V3" (ekkoxiao.github.io), section "YaRN 扩展": the j-th 2-D pair at
// position m turns by phi = m * theta_j.  Here theta_j = base^(-2j/64) (base
// 10000), the pair is (x_{2j}, x_{2j+1}) and the rotation is counter-clockwise:
//   (x, y) -> (x cos phi - y sin phi, x sin phi + y cos phi).
// "Multi-Head Latent Attention / KeyValue" applies it to the shared key k^R at
// the key's own position, "Query" to every head's q^R at the query position.
//
// One thread rotates 4 pairs (16 bytes) of every head of a row in turn (up
// to 16 heads).  The angle m * theta_j is formed and
// reduced modulo 2 pi in fp64 (positions reach 2^17 and beyond, where an fp32
// product would already be off by ~1e-2 rad); sin/cos of the reduced angle and
// the rotation itself are fp32; the result is rounded to bf16.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace mla {

struct RopeTheta {
  double theta[32];  // theta_j = base^(-2j/64), computed on the host in fp64
};

enum : int { kPosExplicit = 0, kPosQuery = 1, kPosCache = 2 };

// Rotate the 4 interleaved pairs (16 bytes) at pairs part*4 .. part*4+3 of a
// 64-element row sitting at position `pos`.
__device__ __forceinline__ uint4 rope_rotate4(uint4 v, int64_t pos, int part, const RopeTheta& th) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = part * 4 + k;
    const double a = (double)pos * th.theta[j];
    const double r = fma(-rint(a * inv_two_pi), two_pi, a);
    float sn, cs;
    sincosf((float)r, &sn, &cs);
    __nv_bfloat162 pr = *reinterpret_cast<__nv_bfloat162*>(&w[k]);
    const float x = __low2float(pr), y = __high2float(pr);
    const float xo = x * cs - y * sn;
    const float yo = x * sn + y * cs;
    __nv_bfloat162 o = __floats2bfloat162_rn(xo, yo);
    w[k] = *reinterpret_cast<uint32_t*>(&o);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}


// cos and sin of the angles of pairs part*4 .. part*4+3 at position `pos`
// (the angle reduced modulo 2 pi in fp64, as in rope_rotate4).
__device__ __forceinline__ void rope_angles4(int64_t pos, int part, const RopeTheta& th, float (&cs)[4],
                                             float (&sn)[4]) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const double a = (double)pos * th.theta[part * 4 + k];
    const double r = fma(-rint(a * inv_two_pi), two_pi, a);
    sincosf((float)r, &sn[k], &cs[k]);
  }
}

__device__ __forceinline__ uint4 rope_turn4(uint4 v, const float (&cs)[4], const float (&sn)[4]) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 pr = *reinterpret_cast<__nv_bfloat162*>(&w[k]);
    const float x = __low2float(pr), y = __high2float(pr);
    __nv_bfloat162 o = __floats2bfloat162_rn(x * cs[k] - y * sn[k], x * sn[k] + y * cs[k]);
    w[k] = *reinterpret_cast<uint32_t*>(&o);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

constexpr int kRopeHeads = 16;  // heads per thread: the angles are formed once for all of them

// One thread: 4 pairs (16 bytes) of row n for up to kRopeHeads heads, which
// share the row's position and hence its angles.
__global__ void __launch_bounds__(256) rope_kernel(const __nv_bfloat16* __restrict__ x_in,
                                                   int64_t in_sn, int64_t in_sh,
                                                   __nv_bfloat16* __restrict__ x_out,
                                                   int64_t out_sn, int64_t out_sh, int64_t N,
                                                   int nh, int pos_mode,
                                                   const int32_t* __restrict__ pos_src, int group,
                                                   const RopeTheta th) {
  const int nhc = (nh + kRopeHeads - 1) / kRopeHeads;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= N * nhc * 8) return;
  const int part = (int)(tid & 7);
  const int64_t rc = tid >> 3;
  const int64_t n = rc / nhc;
  const int hc = (int)(rc - n * nhc);

  int64_t pos;
  if (pos_mode == kPosExplicit) {
    pos = pos_src[n];
  } else if (pos_mode == kPosQuery) {
    const int64_t b = n / group;
    const int s = (int)(n - b * group);
    pos = (int64_t)pos_src[b] - group + s;
    if (pos < 0) return;
  } else {
    const int64_t b = n / group;
    const int64_t j = n - b * group;
    if (j >= pos_src[b]) return;
    pos = j;
  }

  float cs[4], sn[4];
  rope_angles4(pos, part, th, cs, sn);
  const int h1 = min(nh, (hc + 1) * kRopeHeads);
  for (int hd = hc * kRopeHeads; hd < h1; ++hd) {
    const uint4 v = *reinterpret_cast<const uint4*>(x_in + n * in_sn + hd * in_sh + part * 8);
    *reinterpret_cast<uint4*>(x_out + n * out_sn + hd * out_sh + part * 8) = rope_turn4(v, cs, sn);
  }
}

}  // namespace mla
