// mla_api.cu -- the C ABI declared in include/mla.h: argument validation,
// TMA tensor-map encoding, per-device launch configuration and the launches.
// No call allocates device memory or synchronises (except mla_read_status).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include "mla.h"

#include "absorb.cuh"
#include "append.cuh"
#include "combine_up.cuh"
#include "decode.cuh"
#include "expand.cuh"
#include "prefill.cuh"
#include "rope.cuh"
#include "splitkv.cuh"
#include "up_project.cuh"
#include "wgemm.cuh"

namespace {

// Status word of the kernels that take no workspace (absorb, up-projection).
__device__ uint32_t g_kernel_status;

constexpr uint64_t kTimeoutNs = 1000000000ull;  // bounded waits give up after 1 s
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int max_clusters = 0;       // co-resident 2-CTA decode clusters
  uint32_t* kernel_status = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

#ifdef MLA_DECODE_TRACE
unsigned long long* g_decode_trace = nullptr;  // diagnostic build only: timeline buffer
#endif
#ifdef MLA_PREFILL_TRACE
unsigned long long* g_prefill_trace = nullptr;  // diagnostic build only: timeline buffer
#endif

// Test hook (mla_debug_decode_stall): the wait limit of the next mla_decode
// call whose plan barrier is left incomplete; 0 = none pending.
std::atomic<uint64_t> g_stall_ns{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device set-up: kernel attributes, decode cluster occupancy, status symbol.
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (d.ready) return &d;
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return nullptr;
  if (cudaFuncSetAttribute(mla::decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           mla::kDecSmem) != cudaSuccess ||
      cudaFuncSetAttribute(mla::decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) !=
          cudaSuccess ||
      cudaFuncSetAttribute(mla::absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::absorb_smem_bytes(256)) != cudaSuccess ||
      cudaFuncSetAttribute(mla::up_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::up_smem_bytes(64)) != cudaSuccess ||
      cudaFuncSetAttribute(mla::combine_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::cu_smem_bytes(mla::kCUTile)) != cudaSuccess ||
      cudaFuncSetAttribute(mla::append_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::app_smem_bytes(256)) != cudaSuccess ||
      cudaFuncSetAttribute(mla::wgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::wg_smem_bytes(mla::kWgMaxTile)) != cudaSuccess ||
      cudaFuncSetAttribute(mla::prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::kPfSmem) != cudaSuccess ||
      cudaFuncSetAttribute(mla::expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mla::kExSmem) != cudaSuccess)
    return nullptr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * d.num_sms);
  cfg.blockDim = dim3(mla::kDecThreads);
  cfg.dynamicSmemBytes = mla::kDecSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla::decode_kernel, &cfg) != cudaSuccess ||
      clusters < 1)
    return nullptr;
  d.max_clusters = clusters;
  void* sym = nullptr;
  if (cudaGetSymbolAddress(&sym, g_kernel_status) != cudaSuccess) return nullptr;
  d.kernel_status = static_cast<uint32_t*>(sym);
  d.ready = true;
  return &d;
}

bool encode_tiled(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                  const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                  strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the decode kernel: the score CTA reads 128-row boxes of c
// and q_cat (four 64-column blocks, 64 KB) and of k^R and q^R (16 KB), the
// value CTA 32-row boxes of c (all eight blocks, 32 KB); a block is 64
// columns = 128 bytes, one 128-byte-swizzle atom.
struct DecodeMaps {
  CUtensorMap c0, kr, q, qr, c1;
};

// c_kv and q_cat rows are also seen as [rows][blocks of 64 columns] so that
// one 3-D box brings several 128-byte-swizzle atoms at once: an SM's TMA unit
// sustains a few boxes per microsecond, so large boxes are what reach HBM
// bandwidth.
bool encode_decode_maps(DecodeMaps* m, const void* q_cat, const void* c_kv, const void* k_r,
                        int B, int S, int H, int Lmax) {
  const cuuint64_t rows = (cuuint64_t)B * Lmax, qrows = (cuuint64_t)B * S * H;
  const cuuint64_t c3d[3] = {64, rows, 8}, c3s[2] = {1024, 128};
  const cuuint32_t c0b[3] = {64, (cuuint32_t)mla::kTok, (cuuint32_t)(mla::kCStage / mla::kBlk0)};
  const cuuint32_t c1b[3] = {64, (cuuint32_t)mla::kSub, 8};
  const cuuint64_t kd[2] = {64, rows}, ks[1] = {128};
  const cuuint32_t b2[2] = {64, (cuuint32_t)mla::kTok};
  const cuuint64_t q3d[3] = {64, qrows, 9}, q3s[2] = {1152, 128};
  const cuuint64_t qd[2] = {576, qrows}, qs[1] = {1152};
  return encode_tiled(&m->c0, c_kv, 3, c3d, c3s, c0b) && encode_tiled(&m->kr, k_r, 2, kd, ks, b2) &&
         encode_tiled(&m->q, q_cat, 3, q3d, q3s, c0b) && encode_tiled(&m->qr, q_cat, 2, qd, qs, b2) &&
         encode_tiled(&m->c1, c_kv, 3, c3d, c3s, c1b);
}

// Workspace layout of mla_decode / mla_splitkv_combine.
struct WsLayout {
  int n_rb = 0, G = 0, slots = 0;
  size_t prefix = 0, gfirst = 0, segbase = 0, ml = 0, opart = 0, oexp = 0, total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int B, int S, int H, int max_clusters) {
  WsLayout w;
  w.n_rb = (S * H + 127) / 128;
  w.G = max_clusters / w.n_rb;
  if (w.G < 1) w.G = 1;
  w.slots = w.G + B;  // every group boundary inside a sequence adds one segment
  size_t off = 256;   // [0] sticky device status, [1] plan_ok
  w.prefix = off;  off = align256(off + sizeof(int32_t) * (B + 1));
  w.gfirst = off;  off = align256(off + sizeof(int32_t) * B);
  w.segbase = off; off = align256(off + sizeof(int32_t) * (B + 1));
  w.ml = off;      off = align256(off + sizeof(float) * 2 * (size_t)w.slots * w.n_rb * 128);
  w.opart = off;   off = align256(off + sizeof(uint16_t) * (size_t)w.slots * w.n_rb * 128 * 512);
  w.oexp = off;    off = align256(off + (size_t)w.slots * w.n_rb * 128 * 2);
  w.total = off;
  return w;
}

bool decode_shape_ok(int B, int S, int H) {
  return B >= 1 && S >= 1 && H >= 1 && H <= 128 && S * H <= 2048 && B <= (1 << 20);
}

mla_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// Launch with cudaLaunchKernelEx: optional 2-CTA cluster and optional
// programmatic dependent launch (the kernel may start while the previous
// kernel on the stream finishes; the kernels order themselves with
// griddepcontrol.wait, see sm100.cuh).
template <typename... KArgs, typename... Args>
mla_status launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool pdl, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

extern "C" {

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_BAD_SEQLEN: return "MLA_ERR_BAD_SEQLEN";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_version(void) { return 100; }

#ifdef MLA_PREFILL_TRACE
// Diagnostic build only: device buffer of 8-byte stamps [8][8][128], filled by
// later mla_prefill_attention calls.
void mla_debug_set_prefill_trace(void* device_buffer) {
  g_prefill_trace = static_cast<unsigned long long*>(device_buffer);
}
#endif

#ifdef MLA_DECODE_TRACE
// Diagnostic build only: device buffer of 8-byte stamps,
// [clusters][kTraceEvents][kTraceSlots], filled by later mla_decode calls.
void mla_debug_set_decode_trace(void* device_buffer) {
  g_decode_trace = static_cast<unsigned long long*>(device_buffer);
}
#endif

}  // extern "C"

namespace {

// Shared body of mla_absorb_q and mla_absorb_rope_q (q_rope == nullptr: no RoPE).
mla_status absorb_launch(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* W_UK,
                         const int32_t* seqlens, mla_bf16* q_cat, int B, int S, int H,
                         const mla::RopeTheta& th, void* stream) {
  if (!q_nope || !W_UK || !q_cat || !aligned16(q_nope) || !aligned16(W_UK) || !aligned16(q_cat))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (H > 128) return MLA_ERR_UNSUPPORTED;
  const long long BS = (long long)B * S;
  if (BS > 65535LL * 256) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const int n_tile = BS >= 256 ? 256 : (int)((BS + 15) / 16 * 16);
  CUtensorMap tw, tq;
  // W_UK [H*128 d-rows][512 k] seen as [64 k][H*128 rows][8 k-blocks]: one box = 2 atoms
  const cuuint64_t wd[3] = {64, (cuuint64_t)H * 128, 8};
  const cuuint64_t ws[2] = {1024, 128};
  const cuuint32_t wb[3] = {64, 128, 2};
  const cuuint64_t qd[3] = {128, (cuuint64_t)H, (cuuint64_t)BS};
  const cuuint64_t qs[2] = {256, (cuuint64_t)H * 256};
  const cuuint32_t qb[3] = {64, 1, (cuuint32_t)n_tile};
  if (!encode_tiled(&tw, W_UK, 3, wd, ws, wb) || !encode_tiled(&tq, q_nope, 3, qd, qs, qb))
    return MLA_ERR_INVALID_ARG;
  mla::AbsorbParams p;
  p.q_cat = reinterpret_cast<__nv_bfloat16*>(q_cat);
  p.q_rope = reinterpret_cast<const __nv_bfloat16*>(q_rope);
  p.seqlens = seqlens;
  p.BS = (int)BS;
  p.S = S;
  p.H = H;
  p.n_tile = n_tile;
  p.tmem_cols = pow2_at_least((uint32_t)(2 * n_tile));
  p.status = dev->kernel_status;
  p.timeout_ns = kTimeoutNs;
  const dim3 grid(H, 2, (unsigned)((BS + n_tile - 1) / n_tile));
  mla::absorb_kernel<<<grid, mla::kAbsorbThreads, mla::absorb_smem_bytes(n_tile),
                       (cudaStream_t)stream>>>(tw, tq, p, th);
  return launch_status();
}

// theta_j = base^(-2j/64)
mla::RopeTheta base_theta(double base) {
  mla::RopeTheta th;
  for (int j = 0; j < 32; ++j) th.theta[j] = std::pow(base, -2.0 * j / 64.0);
  return th;
}

// Caller-given frequencies: finite and positive.
bool copy_theta(const double* theta, mla::RopeTheta* th) {
  if (!theta) return false;
  for (int j = 0; j < 32; ++j) {
    if (!(theta[j] > 0.0) || !std::isfinite(theta[j])) return false;
    th->theta[j] = theta[j];
  }
  return true;
}

// mla_rope_apply with the frequencies already formed.
mla_status rope_launch(const mla_bf16* x_in, int64_t in_stride_n, int64_t in_stride_h,
                       mla_bf16* x_out, int64_t out_stride_n, int64_t out_stride_h, int64_t N,
                       int nh, int pos_mode, const int32_t* pos_src, int group,
                       const mla::RopeTheta& th, void* stream) {
  if (!x_in || !x_out || !pos_src || !aligned16(x_in) || !aligned16(x_out)) return MLA_ERR_INVALID_ARG;
  if (N < 0 || nh < 1) return MLA_ERR_INVALID_ARG;
  if ((in_stride_n | in_stride_h | out_stride_n | out_stride_h) & 7) return MLA_ERR_INVALID_ARG;
  if (in_stride_n < 0 || in_stride_h < 0 || out_stride_n < 0 || out_stride_h < 0)
    return MLA_ERR_INVALID_ARG;
  if (pos_mode != mla::kPosExplicit && pos_mode != mla::kPosQuery && pos_mode != mla::kPosCache)
    return MLA_ERR_INVALID_ARG;
  if (pos_mode != mla::kPosExplicit && group < 1) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  const long long threads = N * (long long)((nh + mla::kRopeHeads - 1) / mla::kRopeHeads) * 8;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  mla::rope_kernel<<<(unsigned)grid, block, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const __nv_bfloat16*>(x_in), in_stride_n, in_stride_h,
      reinterpret_cast<__nv_bfloat16*>(x_out), out_stride_n, out_stride_h, N, nh, pos_mode,
      pos_src, group, th);
  return launch_status();
}

}  // namespace

extern "C" {

mla_status mla_absorb_q(const mla_bf16* q_nope, const mla_bf16* W_UK, mla_bf16* q_cat, int B,
                        int S, int H, void* stream) {
  return absorb_launch(q_nope, nullptr, W_UK, nullptr, q_cat, B, S, H, base_theta(10000.0), stream);
}

mla_status mla_absorb_rope_q(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* W_UK,
                             const int32_t* seqlens, mla_bf16* q_cat, int B, int S, int H,
                             float base, void* stream) {
  if (!q_rope || !seqlens || !aligned16(q_rope)) return MLA_ERR_INVALID_ARG;
  if (!(base > 1.0f) || !std::isfinite(base)) return MLA_ERR_INVALID_ARG;
  return absorb_launch(q_nope, q_rope, W_UK, seqlens, q_cat, B, S, H, base_theta(base), stream);
}

mla_status mla_absorb_rope_q_freq(const mla_bf16* q_nope, const mla_bf16* q_rope,
                                  const mla_bf16* W_UK, const int32_t* seqlens, mla_bf16* q_cat,
                                  int B, int S, int H, const double* theta, void* stream) {
  if (!q_rope || !seqlens || !aligned16(q_rope)) return MLA_ERR_INVALID_ARG;
  mla::RopeTheta th;
  if (!copy_theta(theta, &th)) return MLA_ERR_INVALID_ARG;
  return absorb_launch(q_nope, q_rope, W_UK, seqlens, q_cat, B, S, H, th, stream);
}

int mla_rope_yarn_frequencies(double base, double s, double alpha, double beta, double orig_len,
                              double* theta) {
  if (!theta || !(base > 1.0) || !std::isfinite(base) || !(s >= 1.0) || !std::isfinite(s) ||
      !(beta > alpha) || !std::isfinite(alpha) || !std::isfinite(beta) || !(orig_len > 0.0) ||
      !std::isfinite(orig_len))
    return MLA_ERR_INVALID_ARG;
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = 0; j < 32; ++j) {
    const double th = std::pow(base, -2.0 * j / 64.0);
    // blend weight: 0 below alpha turns over the original context, 1 above beta
    const double turns = orig_len * th / two_pi;
    const double w = std::min(1.0, std::max(0.0, (turns - alpha) / (beta - alpha)));
    theta[j] = w * th + (1.0 - w) * (th / s);
  }
  return MLA_OK;
}

int mla_rope_yarn_softmax_scale(double s, double* scale) {
  if (!scale || !(s >= 1.0) || !std::isfinite(s)) return MLA_ERR_INVALID_ARG;
  *scale = (0.1 * std::log(s) + 1.0) / std::sqrt((double)(MLA_D_H + MLA_D_R));
  return MLA_OK;
}

mla_status mla_rope_apply(const mla_bf16* x_in, int64_t in_stride_n, int64_t in_stride_h,
                          mla_bf16* x_out, int64_t out_stride_n, int64_t out_stride_h, int64_t N,
                          int nh, int pos_mode, const int32_t* pos_src, int group, float base,
                          void* stream) {
  if (!(base > 1.0f) || !std::isfinite(base)) return MLA_ERR_INVALID_ARG;
  return rope_launch(x_in, in_stride_n, in_stride_h, x_out, out_stride_n, out_stride_h, N, nh,
                     pos_mode, pos_src, group, base_theta(base), stream);
}

mla_status mla_rope_apply_freq(const mla_bf16* x_in, int64_t in_stride_n, int64_t in_stride_h,
                               mla_bf16* x_out, int64_t out_stride_n, int64_t out_stride_h,
                               int64_t N, int nh, int pos_mode, const int32_t* pos_src, int group,
                               const double* theta, void* stream) {
  mla::RopeTheta th;
  if (!copy_theta(theta, &th)) return MLA_ERR_INVALID_ARG;
  return rope_launch(x_in, in_stride_n, in_stride_h, x_out, out_stride_n, out_stride_h, N, nh,
                     pos_mode, pos_src, group, th, stream);
}

size_t mla_decode_workspace_size(int B, int S, int H) {
  if (!decode_shape_ok(B, S, H)) return 0;
  const DeviceInfo* dev = device_info();
  if (!dev) return 0;
  return ws_layout(B, S, H, dev->max_clusters).total;
}

mla_status mla_decode(const mla_bf16* q_cat, const mla_bf16* c_kv, const mla_bf16* k_r,
                      const int32_t* seqlens, int B, int S, int H, int Lmax, float softmax_scale,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!q_cat || !c_kv || !k_r || !seqlens || !aligned16(q_cat) || !aligned16(c_kv) ||
      !aligned16(k_r))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Lmax < 1 || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  if (!decode_shape_ok(B, S, H)) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * Lmax + mla::kTok > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLA_ERR_WORKSPACE;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const WsLayout w = ws_layout(B, S, H, dev->max_clusters);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = (cudaStream_t)stream;

  DecodeMaps maps;
  if (!encode_decode_maps(&maps, q_cat, c_kv, k_r, B, S, H, Lmax)) return MLA_ERR_INVALID_ARG;

  mla::DecodeParams p;
  p.seqlens = seqlens;
  p.prefix = reinterpret_cast<int32_t*>(ws + w.prefix);
  p.gfirst = reinterpret_cast<int32_t*>(ws + w.gfirst);
  p.segbase = reinterpret_cast<int32_t*>(ws + w.segbase);
  p.ml = reinterpret_cast<float2*>(ws + w.ml);
  p.opart = reinterpret_cast<uint4*>(ws + w.opart);
  p.oexp = ws + w.oexp;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.plan_ok = reinterpret_cast<uint32_t*>(ws) + 1;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Lmax = Lmax;
  p.n_rb = w.n_rb;
  p.G = w.G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.timeout_ns = kTimeoutNs;
  p.plan_arrivals = 1u;
  if (const uint64_t stall = g_stall_ns.exchange(0)) {
    p.plan_arrivals = 2u;
    p.timeout_ns = stall;
  }
#ifdef MLA_DECODE_TRACE
  p.trace = g_decode_trace;
#else
  p.trace = nullptr;
#endif

  return launch_ex(mla::decode_kernel, dim3(2 * w.G * w.n_rb), dim3(mla::kDecThreads), mla::kDecSmem,
                   st, true, 2, maps.c0, maps.kr, maps.q, maps.qr, maps.c1, p);
}


mla_status mla_splitkv_combine(const void* workspace, size_t workspace_bytes, mla_bf16* o_lat,
                               int B, int S, int H, void* stream) {
  if (!o_lat || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (!decode_shape_ok(B, S, H)) return MLA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLA_ERR_WORKSPACE;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const WsLayout w = ws_layout(B, S, H, dev->max_clusters);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  mla::CombineParams p;
  p.prefix = reinterpret_cast<const int32_t*>(ws + w.prefix);
  p.gfirst = reinterpret_cast<const int32_t*>(ws + w.gfirst);
  p.segbase = reinterpret_cast<const int32_t*>(ws + w.segbase);
  p.ml = reinterpret_cast<const float2*>(ws + w.ml);
  p.opart = reinterpret_cast<const uint4*>(ws + w.opart);
  p.oexp = ws + w.oexp;
  p.o_lat = reinterpret_cast<__nv_bfloat16*>(o_lat);
  p.plan_ok = reinterpret_cast<const uint32_t*>(ws) + 1;
  p.B = B;
  p.S = S;
  p.H = H;
  p.n_rb = w.n_rb;
  p.G = w.G;
  const dim3 grid((unsigned)(B * w.n_rb), 512 / mla::kCombineCols);
  return launch_ex(mla::combine_kernel, grid, dim3(128), 0, (cudaStream_t)stream, true, 1, p);
}

mla_status mla_up_project(const mla_bf16* o_lat, const mla_bf16* W_UV, mla_bf16* out, int B,
                          int S, int H, void* stream) {
  if (!o_lat || !W_UV || !out || !aligned16(o_lat) || !aligned16(W_UV) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (H > 128) return MLA_ERR_UNSUPPORTED;
  const long long BS = (long long)B * S;
  if (BS > 65535LL * 64) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const int n_tile = BS >= 64 ? 64 : (int)((BS + 15) / 16 * 16);
  CUtensorMap tw, to;
  // W_UV [H*128 v-rows][512 k] seen as [64 k][H*128 rows][8 k-blocks]: one box = 2 atoms
  const cuuint64_t wd[3] = {64, (cuuint64_t)H * 128, 8};
  const cuuint64_t ws[2] = {1024, 128};
  const cuuint32_t wb[3] = {64, 128, 2};
  // o_lat [BS][H][512] seen as [64 k][BS][8 k-blocks][H]: one box = all 8 atoms of n_tile rows
  const cuuint64_t od[4] = {64, (cuuint64_t)BS, 8, (cuuint64_t)H};
  const cuuint64_t os[3] = {(cuuint64_t)H * 1024, 128, 1024};
  const cuuint32_t ob[4] = {64, (cuuint32_t)n_tile, 8, 1};
  if (!encode_tiled(&tw, W_UV, 3, wd, ws, wb) || !encode_tiled(&to, o_lat, 4, od, os, ob))
    return MLA_ERR_INVALID_ARG;
  mla::UpParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.BS = (int)BS;
  p.H = H;
  p.n_tile = n_tile;
  p.tmem_cols = pow2_at_least((uint32_t)n_tile);
  p.status = dev->kernel_status;
  p.timeout_ns = kTimeoutNs;
  const dim3 grid(H, (unsigned)((BS + n_tile - 1) / n_tile));
  return launch_ex(mla::up_project_kernel, grid, dim3(mla::kUpThreads), mla::up_smem_bytes(n_tile),
                   (cudaStream_t)stream, true, 1, tw, to, p);
}

mla_status mla_combine_up_project(const void* workspace, size_t workspace_bytes, const mla_bf16* W_UV,
                                  mla_bf16* out, int B, int S, int H, void* stream) {
  if (!W_UV || !out || !aligned16(W_UV) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (!decode_shape_ok(B, S, H)) return MLA_ERR_UNSUPPORTED;
  const long long BS = (long long)B * S;
  if (BS > 65535LL * mla::kCUTile) return MLA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLA_ERR_WORKSPACE;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const WsLayout w = ws_layout(B, S, H, dev->max_clusters);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
  if (w.G > 32 * mla::kCUSegLanes) return MLA_ERR_UNSUPPORTED;  // more segments per row than lanes hold
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const int n_tile = BS >= mla::kCUTile ? mla::kCUTile : (int)((BS + 15) / 16 * 16);
  CUtensorMap tw;
  // W_UV [H*128 v-rows][512 k] seen as [64 k][H*128 rows][8 k-blocks]: one box = 2 atoms
  const cuuint64_t wd[3] = {64, (cuuint64_t)H * 128, 8};
  const cuuint64_t wst[2] = {1024, 128};
  const cuuint32_t wb[3] = {64, 128, 2};
  if (!encode_tiled(&tw, W_UV, 3, wd, wst, wb)) return MLA_ERR_INVALID_ARG;
  mla::CombineUpParams p;
  p.prefix = reinterpret_cast<const int32_t*>(ws + w.prefix);
  p.gfirst = reinterpret_cast<const int32_t*>(ws + w.gfirst);
  p.segbase = reinterpret_cast<const int32_t*>(ws + w.segbase);
  p.ml = reinterpret_cast<const float2*>(ws + w.ml);
  p.opart = reinterpret_cast<const uint4*>(ws + w.opart);
  p.oexp = ws + w.oexp;
  p.plan_ok = reinterpret_cast<const uint32_t*>(ws) + 1;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.B = B;
  p.S = S;
  p.H = H;
  p.n_rb = w.n_rb;
  p.G = w.G;
  p.BS = (int)BS;
  p.n_tile = n_tile;
  p.tmem_cols = pow2_at_least((uint32_t)n_tile);
  p.status = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(ws));
  p.timeout_ns = kTimeoutNs;
  const dim3 grid(H, (unsigned)((BS + n_tile - 1) / n_tile));
  return launch_ex(mla::combine_up_kernel, grid, dim3(mla::kCUTile * 32), mla::cu_smem_bytes(n_tile),
                   (cudaStream_t)stream, true, 1, tw, p);
}

size_t mla_cache_append_workspace_size(int B, int S, int d) {
  if (B < 1 || S < 1 || d < 64 || (d & 63) != 0) return 0;
  const size_t ks = (size_t)(d + mla::kAppKc - 1) / mla::kAppKc;
  return 256 + align256(sizeof(float) * ks * (size_t)B * S * mla::kAppCols);
}

mla_status mla_cache_append(const mla_bf16* h, const mla_bf16* W_DKV, const mla_bf16* W_KR,
                            const int32_t* seqlens, mla_bf16* c_kv, mla_bf16* k_r, int B, int S, int d,
                            int Lmax, const double* theta, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!h || !W_DKV || !W_KR || !seqlens || !c_kv || !k_r || !aligned16(h) || !aligned16(W_DKV) ||
      !aligned16(W_KR) || !aligned16(c_kv) || !aligned16(k_r))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Lmax < S || d < 64) return MLA_ERR_INVALID_ARG;
  if ((d & 63) != 0 || d > (1 << 20)) return MLA_ERR_UNSUPPORTED;
  const long long BS = (long long)B * S;
  if (BS > 65535LL * 256 || (long long)B * Lmax > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLA_ERR_WORKSPACE;
  if (workspace_bytes < mla_cache_append_workspace_size(B, S, d)) return MLA_ERR_WORKSPACE;
  mla::RopeTheta th = base_theta(10000.0);
  if (theta && !copy_theta(theta, &th)) return MLA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const int ks = (d + mla::kAppKc - 1) / mla::kAppKc;
  const int n_tile = BS >= 256 ? 256 : (int)((BS + 15) / 16 * 16);
  // row-major [rows][d] seen as [64 columns][rows][d / 64 atoms]: one box = four
  // 128-byte-swizzle atoms of 128 (weights) or n_tile (tokens) rows
  const cuuint64_t nat = (cuuint64_t)(d / 64);
  const cuuint64_t str[2] = {(cuuint64_t)d * 2, 128};
  const cuuint64_t dd[3] = {64, 512, nat}, dr[3] = {64, 64, nat}, dh[3] = {64, (cuuint64_t)BS, nat};
  const cuuint32_t bw[3] = {64, 128, 4}, bh[3] = {64, (cuuint32_t)n_tile, 4};
  CUtensorMap twd, twr, th_map;
  if (!encode_tiled(&twd, W_DKV, 3, dd, str, bw) || !encode_tiled(&twr, W_KR, 3, dr, str, bw) ||
      !encode_tiled(&th_map, h, 3, dh, str, bh))
    return MLA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  mla::AppendParams p;
  p.part = reinterpret_cast<float*>(ws + 256);
  p.BS = (int)BS;
  p.n_tile = n_tile;
  p.ks = ks;
  p.tmem_cols = pow2_at_least((uint32_t)n_tile);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.timeout_ns = kTimeoutNs;
  p.barrier = reinterpret_cast<uint32_t*>(ws) + 1;  // words 1 (arrivals) and 2 (generation)
  mla::AppendFinalizeParams& f = p.fin;
  f.part = p.part;
  f.seqlens = seqlens;
  f.c_kv = reinterpret_cast<__nv_bfloat16*>(c_kv);
  f.k_r = reinterpret_cast<__nv_bfloat16*>(k_r);
  f.status = p.status;
  f.BS = (int)BS;
  f.S = S;
  f.ks = ks;
  f.Lmax = Lmax;
  cudaStream_t st = (cudaStream_t)stream;
  const dim3 grid(5, (unsigned)ks, (unsigned)((BS + n_tile - 1) / n_tile));
  const size_t smem = mla::app_smem_bytes(n_tile);
  // One cooperative launch (the finalize after a grid-wide barrier) when every
  // CTA can be resident at once; otherwise the GEMM and the finalize kernel.
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mla::append_gemm_kernel, mla::kAppThreads, smem) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  const long long ctas = 5LL * ks * grid.z;
  if (ctas <= (long long)per_sm * dev->num_sms) {
    p.fused = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(mla::kAppThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::append_gemm_kernel, twd, twr, th_map, p, th) != cudaSuccess)
      return MLA_ERR_CUDA;
    return launch_status();
  }
  p.fused = 0;
  const mla_status s1 = launch_ex(mla::append_gemm_kernel, grid, dim3(mla::kAppThreads), smem, st, true, 1, twd,
                                  twr, th_map, p, th);
  if (s1 != MLA_OK) return s1;
  return launch_ex(mla::append_finalize_kernel, dim3((unsigned)BS), dim3(mla::kAppCols / 2), 0, st, true, 1,
                   p.fin, th);
}

mla_status mla_debug_decode_stall(uint64_t wait_limit_ns) {
  if (wait_limit_ns == 0 || wait_limit_ns > kTimeoutNs) return MLA_ERR_INVALID_ARG;
  g_stall_ns.store(wait_limit_ns);
  return MLA_OK;
}

}  // extern "C"

namespace {

// Launch shape of the output projection: token tiles of up to 64, weight
// tiles of 128 rows, and ks near-equal slices of K so that the grid fills the
// SMs two CTAs deep.
struct WgPlan {
  int n_tile = 0, ntiles = 0, mtiles = 0, total_chunks = 0, ks = 1;
  size_t ws = 0;
};

WgPlan wg_plan(int BS, int K, int d, int num_sms) {
  WgPlan w;
  w.n_tile = BS >= mla::kWgMaxTile ? mla::kWgMaxTile : (BS + 15) / 16 * 16;
  w.ntiles = (BS + w.n_tile - 1) / w.n_tile;
  w.mtiles = d / 128;
  w.total_chunks = K / mla::kWgKc;
  const long long tiles = (long long)w.mtiles * w.ntiles;
  w.ks = (int)std::max(1LL, std::min((long long)w.total_chunks, 2LL * num_sms / std::max(1LL, tiles)));
  w.ws = w.ks > 1 ? sizeof(float) * (size_t)w.ks * BS * d : 0;
  return w;
}

bool wg_shape_ok(int BS, int K, int d) {
  return BS >= 1 && K >= mla::kWgKc && d >= 128 && K % mla::kWgKc == 0 && d % 128 == 0 &&
         (long long)BS <= 65535LL * mla::kWgMaxTile && (long long)d / 128 <= 0x7fffffffLL && K <= (1 << 24);
}

// u = W x through wgemm_kernel (and the slice reduction when w.ks > 1).
mla_status wg_launch(const mla_bf16* x, const mla_bf16* W, mla_bf16* u, int BS, int K, int d, const WgPlan& w,
                     const DeviceInfo* dev, void* workspace, void* stream) {
  // row-major [rows][K] seen as [64 columns][rows][K / 64 atoms]: one box =
  // two 128-byte-swizzle atoms of 128 weight rows or n_tile token rows
  const cuuint64_t str[2] = {(cuuint64_t)K * 2, 128};
  const cuuint64_t dw[3] = {64, (cuuint64_t)d, (cuuint64_t)(K / 64)}, dx[3] = {64, (cuuint64_t)BS, (cuuint64_t)(K / 64)};
  const cuuint32_t bw[3] = {64, 128, 2}, bx[3] = {64, (cuuint32_t)w.n_tile, 2};
  CUtensorMap tw, tx;
  if (!encode_tiled(&tw, W, 3, dw, str, bw) || !encode_tiled(&tx, x, 3, dx, str, bx)) return MLA_ERR_INVALID_ARG;
  mla::WGemmParams p;
  p.part = static_cast<float*>(workspace);
  p.out = reinterpret_cast<__nv_bfloat16*>(u);
  p.BS = BS;
  p.M = d;
  p.n_tile = w.n_tile;
  p.ks = w.ks;
  p.total_chunks = w.total_chunks;
  p.tmem_cols = pow2_at_least((uint32_t)w.n_tile);
  p.status = dev->kernel_status;
  p.timeout_ns = kTimeoutNs;
  cudaStream_t st = (cudaStream_t)stream;
  const mla_status s1 = launch_ex(mla::wgemm_kernel, dim3((unsigned)w.mtiles, (unsigned)w.ks, (unsigned)w.ntiles),
                                  dim3(mla::kWgThreads), mla::wg_smem_bytes(w.n_tile), st, true, 1, tw, tx, p);
  if (s1 != MLA_OK || w.ks == 1) return s1;
  const size_t total4 = (size_t)BS * d / 4;
  return launch_ex(mla::wgemm_reduce_kernel, dim3((unsigned)((total4 + 255) / 256)), dim3(256), 0, st, true, 1,
                   static_cast<const float*>(workspace), reinterpret_cast<__nv_bfloat16*>(u), BS, d, w.ks);
}

}  // namespace

extern "C" {

size_t mla_output_project_workspace_size(int BS, int K, int d) {
  if (!wg_shape_ok(BS, K, d)) return 0;
  const DeviceInfo* dev = device_info();
  if (!dev) return 0;
  return wg_plan(BS, K, d, dev->num_sms).ws;
}

mla_status mla_output_project(const mla_bf16* x, const mla_bf16* W, mla_bf16* u, int BS, int K, int d,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !W || !u || !aligned16(x) || !aligned16(W) || !aligned16(u)) return MLA_ERR_INVALID_ARG;
  if (BS < 1 || K < 1 || d < 1) return MLA_ERR_INVALID_ARG;
  if (!wg_shape_ok(BS, K, d)) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const WgPlan w = wg_plan(BS, K, d, dev->num_sms);
  if (w.ws > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.ws))
    return MLA_ERR_WORKSPACE;
  return wg_launch(x, W, u, BS, K, d, w, dev, workspace, stream);
}

mla_status mla_prefill_expand(const mla_bf16* c_kv, const mla_bf16* W_UK, const mla_bf16* W_UV, mla_bf16* k_c,
                              mla_bf16* v_c, int B, int Lmax, int H, void* stream) {
  if (!c_kv || !W_UK || !W_UV || !k_c || !v_c || !aligned16(c_kv) || !aligned16(W_UK) || !aligned16(W_UV) ||
      !aligned16(k_c) || !aligned16(v_c))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || Lmax < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  const long long rows = (long long)B * Lmax;
  if (H > 128 || rows + 128 > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  // [rows][512] seen as [64 columns][rows][8 atoms]: the latent rows in two
  // boxes of four atoms (64 KB), a weight's 128 rows of one head in boxes of
  // two atoms (32 KB)
  const cuuint64_t str[2] = {1024, 128};
  const cuuint64_t dc[3] = {64, (cuuint64_t)rows, 8}, dw[3] = {64, (cuuint64_t)H * 128, 8};
  const cuuint32_t bc[3] = {64, 128, 4}, bw[3] = {64, 128, 2};
  CUtensorMap tc, tk, tv;
  if (!encode_tiled(&tc, c_kv, 3, dc, str, bc) || !encode_tiled(&tk, W_UK, 3, dw, str, bw) ||
      !encode_tiled(&tv, W_UV, 3, dw, str, bw))
    return MLA_ERR_INVALID_ARG;
  mla::ExpandParams p;
  p.k_c = reinterpret_cast<__nv_bfloat16*>(k_c);
  p.v_c = reinterpret_cast<__nv_bfloat16*>(v_c);
  p.T = (int)rows;
  p.H = H;
  p.n_tt = (int)((rows + 127) / 128);
  p.n_grp = 2 * ((H + mla::kExGroup - 1) / mla::kExGroup);
  p.status = dev->kernel_status;
  p.timeout_ns = kTimeoutNs;
  const long long units = (long long)p.n_tt * p.n_grp;
  const int grid = (int)std::min<long long>(units, dev->num_sms);
  return launch_ex(mla::expand_kernel, dim3((unsigned)grid), dim3(mla::kExThreads), mla::kExSmem,
                   (cudaStream_t)stream, true, 1, tc, tk, tv, p);
}

mla_status mla_prefill_attention(const mla_bf16* q_nope, const mla_bf16* q_rope, const mla_bf16* k_c,
                                 const mla_bf16* k_r, const mla_bf16* v_c, const int32_t* seqlens, int B, int S,
                                 int H, int Lmax, float softmax_scale, mla_bf16* out, void* stream) {
  if (!q_nope || !q_rope || !k_c || !k_r || !v_c || !seqlens || !out || !aligned16(q_nope) || !aligned16(q_rope) ||
      !aligned16(k_c) || !aligned16(k_r) || !aligned16(v_c) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Lmax < 1 || S > Lmax || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  const int nq = (S + 127) / 128;
  if (H > 128 || (long long)B * Lmax + 128 > 0x7fffffffLL || (long long)B * S + 128 > 0x7fffffffLL ||
      (long long)B * H * nq > 0x7fffffffLL)
    return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  // [rows][H][128] seen as [64 columns][rows][2 atoms][H]: one box = the two
  // 128-byte-swizzle atoms of 128 rows of one head; [rows][H][64] and
  // [rows][64] likewise with one atom.
  const cuuint64_t qrows = (cuuint64_t)B * S, krows = (cuuint64_t)B * Lmax, hh = (cuuint64_t)H;
  const cuuint64_t dq[4] = {64, qrows, 2, hh}, dk[4] = {64, krows, 2, hh};
  const cuuint64_t s4[3] = {hh * 256, 128, 256};
  const cuuint64_t dqr[3] = {64, qrows, hh}, sqr[2] = {hh * 128, 128};
  const cuuint64_t dkr[2] = {64, krows}, skr[1] = {128};
  const cuuint32_t b4[4] = {64, 128, 2, 1}, b3[3] = {64, 128, 1}, b2[2] = {64, 128};
  CUtensorMap tqn, tqr, tkc, tkr, tvc;
  if (!encode_tiled(&tqn, q_nope, 4, dq, s4, b4) || !encode_tiled(&tqr, q_rope, 3, dqr, sqr, b3) ||
      !encode_tiled(&tkc, k_c, 4, dk, s4, b4) || !encode_tiled(&tkr, k_r, 2, dkr, skr, b2) ||
      !encode_tiled(&tvc, v_c, 4, dk, s4, b4))
    return MLA_ERR_INVALID_ARG;
  mla::PrefillParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.seqlens = seqlens;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Lmax = Lmax;
  p.nq = nq;
  p.n_units = B * H * ((nq + 1) / 2);
  p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  p.status = dev->kernel_status;
  p.timeout_ns = kTimeoutNs;
#ifdef MLA_PREFILL_TRACE
  p.trace = g_prefill_trace;
#else
  p.trace = nullptr;
#endif
  const int grid = std::min(p.n_units, dev->num_sms);
  return launch_ex(mla::prefill_kernel, dim3((unsigned)grid), dim3(mla::kPfThreads), mla::kPfSmem,
                   (cudaStream_t)stream, true, 1, tqn, tqr, tkc, tkr, tvc, p);
}

mla_status mla_read_status(void* workspace, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  uint32_t bits = 0, kbits = 0;
  if (workspace) {
    if (cudaMemcpy(&bits, workspace, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(workspace, 0, sizeof bits) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (cudaMemcpy(&kbits, dev->kernel_status, sizeof kbits, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dev->kernel_status, 0, sizeof kbits) != cudaSuccess)
    return MLA_ERR_CUDA;
  bits |= kbits;
  if (bits & mla::kDevErrInternal) return MLA_ERR_CUDA;
  if (bits & mla::kDevErrTimeout) return MLA_ERR_TIMEOUT;
  if (bits & mla::kDevErrBadSeqlen) return MLA_ERR_BAD_SEQLEN;
  return MLA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode (mla_decode_noalloc).  For callers that cannot
// allocate device memory on their decode path, the split-KV workspace lives
// in this fixed array instead of a caller buffer.  In host code the name
// g_static_scratch is only a host-side stand-in for the symbol; the device
// address comes from cudaGetSymbolAddress, looked up once per device.
namespace {

__device__ __align__(256) uint8_t g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

std::mutex g_static_mutex;
uint8_t* g_static_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (nullptr on error).
uint8_t* static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_addr[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || addr == nullptr)
      return nullptr;
    g_static_addr[dev] = static_cast<uint8_t*>(addr);
  }
  return g_static_addr[dev];
}

}  // namespace

extern "C" mla_status mla_decode_noalloc(const mla_bf16* q_cat, const mla_bf16* c_kv,
                                         const mla_bf16* k_r, const int32_t* seqlens, int B,
                                         int S, int H, int Lmax, float softmax_scale,
                                         mla_bf16* o_lat, void* stream) {
  if (!q_cat || !c_kv || !k_r || !seqlens || !o_lat || !aligned16(q_cat) || !aligned16(c_kv) ||
      !aligned16(k_r) || !aligned16(o_lat))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Lmax < 1 || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  if (!decode_shape_ok(B, S, H)) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * Lmax + mla::kTok > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (!dev) return MLA_ERR_CUDA;
  const WsLayout w = ws_layout(B, S, H, dev->max_clusters);
  if (w.total > (size_t)MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  uint8_t* ws = static_scratch();
  if (!ws) return MLA_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  // Device errors go to the library status word; word [1] of the scratch is
  // the plan's ok flag, rewritten by the decode kernel on every call.
  uint32_t* status = dev->kernel_status;
  uint32_t* plan_ok = reinterpret_cast<uint32_t*>(ws) + 1;

  DecodeMaps maps;
  if (!encode_decode_maps(&maps, q_cat, c_kv, k_r, B, S, H, Lmax)) return MLA_ERR_INVALID_ARG;

  mla::DecodeParams p;
  p.seqlens = seqlens;
  p.prefix = reinterpret_cast<int32_t*>(ws + w.prefix);
  p.gfirst = reinterpret_cast<int32_t*>(ws + w.gfirst);
  p.segbase = reinterpret_cast<int32_t*>(ws + w.segbase);
  p.ml = reinterpret_cast<float2*>(ws + w.ml);
  p.opart = reinterpret_cast<uint4*>(ws + w.opart);
  p.oexp = ws + w.oexp;
  p.status = status;
  p.plan_ok = plan_ok;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Lmax = Lmax;
  p.n_rb = w.n_rb;
  p.G = w.G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.timeout_ns = kTimeoutNs;
  p.plan_arrivals = 1u;
  p.trace = nullptr;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * w.G * w.n_rb);
  cfg.blockDim = dim3(mla::kDecThreads);
  cfg.dynamicSmemBytes = mla::kDecSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mla::decode_kernel, maps.c0, maps.kr, maps.q, maps.qr, maps.c1, p) !=
      cudaSuccess)
    return MLA_ERR_CUDA;

  mla::CombineParams cp;
  cp.prefix = p.prefix;
  cp.gfirst = p.gfirst;
  cp.segbase = p.segbase;
  cp.ml = p.ml;
  cp.opart = p.opart;
  cp.oexp = p.oexp;
  cp.o_lat = reinterpret_cast<__nv_bfloat16*>(o_lat);
  cp.plan_ok = plan_ok;
  cp.B = B;
  cp.S = S;
  cp.H = H;
  cp.n_rb = w.n_rb;
  cp.G = w.G;
  mla::combine_kernel<<<dim3((unsigned)(B * w.n_rb), 512 / mla::kCombineCols), 128, 0, st>>>(cp);
  return launch_status();
}
