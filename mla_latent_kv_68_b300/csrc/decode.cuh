// decode.cuh -- latent-space MLA decode over the compressed cache, split-KV.
//
// "DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention":
//   score   s_j = (q~ . c_j + q^R . k^R_j) / sqrt(d_h + d_h^R)   ("注意力计算",
//           with the absorbed content term of "潜在向量的作用")
//   softmax over the visible positions, aggregation in latent space
//           o_lat = sum_j a_j c_j                                   ("潜在向量的作用")
// All query rows of one sequence (S*H of them, up to 128 per "row block")
// share every cache tile, so one 128-token tile feeds two dense contractions:
//   S[128 x 128]   = Q[128 x 576] . K_tile[128 x 576]^T      (K = [c ; k^R])
//   O[128 x 512]  += P[128 x 128] . C_tile[128 x 512]
//
// B300 mapping.  A tcgen05 MMA of M = 128 runs at the full tensor rate only
// from N = 128 up (N = 64 reaches about half of it), so both contractions use
// N >= 128.  The fp32 accumulator O (128 x 512) fills one SM's whole tensor
// memory, so each unit of work is a CLUSTER OF TWO CTAs on two SMs:
//   rank 0 ("score CTA"): q~ (128 x 512 bf16) lives in its tensor memory as
//       the A operand of the QK^T MMAs (A-from-TMEM form), next to two
//       128-column S buffers (the MMAs of tile i+1 fill one while the softmax
//       reads tile i from the other); q^R (128 x 64) sits in shared memory.
//       Shared memory is otherwise left to the TMA rings, whose depth sets
//       how many bytes an SM keeps in flight.
//       Operands arrive through two TMA rings: a c ring of 64 KB stages, each
//       one box of four 128-row x 64-column blocks (one 128-byte-swizzle atom
//       per block), and a k^R ring of 16 KB stages; a tile is two c stages and
//       one k^R stage.  At a segment start the 512 q~ columns of the 128
//       query rows pass through the c ring (two stages) and the MMA thread
//       moves them into tensor memory with tcgen05.cp (TMA boxes arrive well
//       before row-wise loads, which wait behind the cache stream in L2);
//       q^R goes to a buffer of its own.  Box size and
//       count matter on B300: an SM's TMA unit handles only a few boxes per
//       microsecond, so 16 KB boxes cap an SM near 50 GB/s, 32 KB boxes near
//       65-95 GB/s and 64 KB boxes near 100-120 GB/s.
//       Eight softmax
//       warps (two threads per query row, 64 tokens each) run the online
//       softmax, write P (bf16, in the swizzled K-major layout the MMA reads)
//       and the per-row rescale exponent into a local staging buffer, and one
//       thread moves it into rank 1 with a single bulk shared-to-shared copy
//       that completes a transaction-counted barrier there.
//   rank 1 ("value CTA"): O lives in all 512 columns of its tensor memory; it
//       streams the 512-wide c rows of the same tiles in 64-token stages (one
//       64 KB box each; L2 hits right after rank 0's reads, so HBM sees every
//       cache byte once) and issues O += P . C with N = 256 and C read as an
//       MN-major operand straight from the TMA tile.
// Neither CTA duplicates the other's tensor work.
//
// Online softmax (log2 domain, s2 = s * scale * log2 e).  Each row keeps an
// INTEGER reference exponent m and l = sum 2^(s2 - m) of the bf16-rounded
// weights it sent.  m moves only when a tile's maximum exceeds m + 8; then
// m := ceil(max) and O, l are scaled by alpha = 2^(m_old - m_new), an exact
// power of two, so the rescale adds no rounding.  Weights stay <= 2^8.
//
// Split-KV: the grid is G groups x (row blocks) clusters; group g owns a
// contiguous run of cache tiles over all sequences (splitkv.cuh).  Each
// segment (a sequence's share of a group's run) leaves O unnormalised plus
// (m, l) per row; splitkv.cuh merges them.
//
// Cold code.  The first pass through the softmax's exponent section (about
// 6 KB of unrolled code) takes about 5 us: its instruction lines miss one
// after another, in step on every SM, with or without the cache stream
// running.  Run on the first tile, that sits on the path every later tile
// waits on.  So it is run early, "dry", on a stand-in tile -- no waits, no
// barrier arrivals, no global reads or writes, results discarded -- by the
// row warps of both CTAs, which are idle then (the first scores and the
// first P arrive several microseconds later).  The dry visit needs nothing
// from the kernels before this one, so it starts before the dependency wait.
// (The softmax is also written as rolled loops over 16-column slices, which
// keeps that first pass short.)
//
// Every wait is bounded (sm100.cuh), including the exchanges between the two
// threads of a row, which go through mbarriers rather than bar.sync.  A wait
// that runs out aborts the CTA's remaining work; the cluster peer notices
// through its own waits.  Both CTAs meet in a final cluster barrier so neither
// exits while the other may still touch its shared memory.
#pragma once

#include "sm100.cuh"
#include "splitkv.cuh"

namespace mla {

constexpr int kDecThreads = 384;  // 12 warps: 0 TMA, 1 MMA, 2 P copy / release, 4..11 rows
constexpr int kTok = kTileRows;   // cache rows per tile (128)
// score CTA (rank 0)
constexpr int kBlk0 = kTok * 128;          // one block: 128 rows x 64 bf16 = 16 KB
constexpr int kCStage = 4 * kBlk0;         // c ring stage: four blocks (one 64 KB TMA box)
constexpr int kCStages = 2;
constexpr int kCPerTile = 2;               // c stages per 128-row tile (512 columns)
constexpr int kRStage = kBlk0;             // k^R ring stage: one block (16 KB)
constexpr int kRStages = 2;
constexpr int kOffR = kCStages * kCStage;  // k^R ring
constexpr int kOffQR = kOffR + kRStages * kRStage;  // q^R of the segment: 128 x 64 bf16 (A of the RoPE MMAs)
constexpr int kOffXch = kOffQR + kBlk0;    // ceil(row max) f32 [2 tiles][2 halves][128], row sum f32 [128]
constexpr int kXchBytes = 2 * 2 * 128 * 4 + 128 * 4;
// a P slot of the value CTA: P (128 x 128 bf16), rescale exponents u32 [128], row sums f32 [128]
constexpr int kPBytes = 128 * kTok * 2;
constexpr int kOffPEx = kPBytes;
constexpr int kOffPL = kOffPEx + 128 * 4;
constexpr uint32_t kPTx = kOffPL + 128 * 4;   // bytes the score CTA stores into one P slot
// value CTA (rank 1)
constexpr int kSub = 32;                   // cache rows per value-CTA stage
constexpr int kBlk1 = kSub * 128;          // 4 KB
constexpr int kStage1 = 8 * kBlk1;         // 32 KB: one TMA box of whole 1 KB rows
constexpr int kStages1 = 5;
constexpr int kStepsPerSub = kSub / 16;    // P . C K-steps per value-CTA stage
constexpr int kOffP = kStages1 * kStage1;  // P slots [2], each P then alpha
// ring barriers of a CTA: the score CTA's c and k^R rings, or the value CTA's ring
constexpr int kRingSlots = (kCStages + kRStages) > kStages1 ? (kCStages + kRStages) : kStages1;
constexpr int kPSlot = 33 * 1024;          // slot stride (keeps P 1 KB aligned)
static_assert(kPTx == (uint32_t)kPSlot, "a P slot is exactly what the score CTA stores into it");
// shared by both
constexpr int kEnd0 = kOffXch + kXchBytes, kEnd1 = kOffP + 2 * kPSlot;
constexpr int kOffBar = kEnd0 > kEnd1 ? kEnd0 : kEnd1;
constexpr int kNumBars = 47;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tensor-memory address, abort flag
constexpr int kOffPlan = kOffMisc + 16;            // PlanState
constexpr int kDecSmem = kOffPlan + 32;
static_assert(kDecSmem <= 232448, "decode shared memory exceeds 227 KB");
static_assert(kRingSlots <= 10, "the FULL / EMPTY barrier ranges hold 10 ring slots each");
static_assert(kOffR % 1024 == 0 && kOffQR % 1024 == 0 && kOffP % 1024 == 0 && kPSlot % 1024 == 0,
              "swizzled operands need 1 KB alignment");
// score CTA tensor memory: S buffers at columns 0..127 and 128..255, q~ at 256..511
constexpr uint32_t kQCol = 256;

// barrier indices
enum : int {
  B_FULL = 0, B_EMPTY = 10,          // TMA rings (rank 0: c, then k^R; rank 1: its c ring), kRingSlots each
  B_SFULL = 20, B_SEMPTY = 22,       // score CTA: the two S buffers
  B_PEMPTY = 24,                     // score CTA: P slot in the value CTA free again
  B_XCH = 26,                        // score CTA: row-max exchange [tile parity][quadrant]
  B_XL = 34,                         // score CTA: row-sum exchange at a segment end
  B_PFULL = 35,                      // value CTA: P + alpha of a tile have arrived
  B_PREADY = 37,                     // value CTA: O rescaled, P may be consumed
  B_PVDONE = 39,                     // value CTA: P . C of a tile completed
  B_OFREE = 41,                      // value CTA: epilogue has read O
  B_DRAIN = 42,                      // both: final MMA drain
  B_QRFULL = 43,                     // score CTA: q^R of the segment has landed
  B_QREMPTY = 44,                    // score CTA: the segment's MMAs no longer read q~ and q^R
  B_PLAN = 45                        // both: the split plan of this CTA's group is in PlanState
};

struct DecodeParams {
  const int32_t* seqlens;      // [B]
  int32_t* prefix;             // plan for the combine (splitkv.cuh), written by CTA 0: [B + 1]
  int32_t* gfirst;             // [B]
  int32_t* segbase;            // [B + 1]
  float2* ml;                  // [slots * n_rb, 128]        (m, l) per row
  uint4* opart;                // [slots * n_rb][64 column octets][128 rows] fp16 x 8: 2^-e O / l per segment
  uint8_t* oexp;               // [slots * n_rb][128 rows][2 column halves]: the exponent e of each half row
  uint32_t* status;
  uint32_t* plan_ok;           // written by CTA 0
  int B, S, H, Lmax, n_rb, G;
  float scale_log2;            // softmax_scale * log2(e)
  uint64_t timeout_ns;
  uint32_t plan_arrivals;      // arrivals that complete the plan barrier: 1 (2 for the stall test hook)
  unsigned long long* trace;   // timeline of a diagnostic build (MLA_DECODE_TRACE), else unused
};

// Diagnostic timeline: with MLA_DECODE_TRACE defined, the kernel stamps the
// global timer at fixed points of each tile into
// trace[cluster][event][tile] (first kTraceSlots tiles or segments).  The
// product build compiles the stamps away.
constexpr int kTraceEvents = 24, kTraceSlots = 64;
enum : int {
  TR_START = 0,       // kernel entry (rank 0, thread 0)           [slot 0]
  TR_PLAN = 1,        // plan ready (rank 0, plan warp)             [slot 0]
  TR_TMA_ISSUE = 2,   // score CTA: first c stage of the tile issued
  TR_QK_BEGIN = 3,    // score CTA: first QK^T MMA of the tile issued
  TR_QK_END = 4,      // score CTA: last QK^T MMA of the tile issued
  TR_S_READY = 5,     // score CTA: a softmax thread saw S
  TR_P_SENT = 6,      // score CTA: that thread has issued its P stores
  TR_P_FULL = 7,      // value CTA: a row thread saw the P slot full
  TR_PV_BEGIN = 8,    // value CTA: first P . C MMA issued
  TR_PV_END = 9,      // value CTA: last P . C MMA issued
  TR_PV_DONE = 10,    // value CTA: P . C completed (releaser)
  TR_EPI_BEGIN = 11,  // value CTA: epilogue of a segment begins      [segment]
  TR_EPI_END = 12,    // value CTA: epilogue stores issued            [segment]
  TR_END = 13,        // wind-down reached (rank 0 / rank 1)          [slot rank]
  TR_V_TMA = 14,      // value CTA: first c stage of the tile issued
  TR_SM_MAX = 15,     // score CTA: that softmax thread has its row maximum
  TR_SM_XCH = 16,     // score CTA: ... and its partner's
  TR_SM_SLOT = 17,    // score CTA: ... and the P slot is free
  TR_QK_LAST = 18,    // score CTA: the tile's last c stage has landed (MMA thread)
  TR_V_LAND = 19      // value CTA: the tile's last c stage has landed (MMA thread)
};
#ifdef MLA_DECODE_TRACE
#define MLA_TRACE(p, ev, idx)                                                                   \
  do {                                                                                          \
    if ((p).trace && (idx) < kTraceSlots)                                                       \
      (p).trace[((size_t)(blockIdx.x >> 1) * kTraceEvents + (ev)) * kTraceSlots + (idx)] =       \
          global_timer_ns();                                                                    \
  } while (0)
#else
#define MLA_TRACE(p, ev, idx) \
  do {                        \
  } while (0)
#endif

struct TileInfo {
  int b, t, L, i, k, slot;
  int nvt;  // cache rows of the sequence inside this tile (1..128)
  bool first, last;
  bool dry;  // warm-up visit of a stand-in tile: compute only, no waits, no global reads or writes
};

// The split plan as one CTA needs it (splitkv.cuh): the total tile count and
// the state of the walk at the sequence holding the group's first tile.
// The split plan lays all sequences end to end in units of work: one unit
// per 128-token tile, after kSeqUnits units that stand for the cost of
// starting a sequence (a cluster that switches to another sequence passes the
// query rows through its ring again and writes one more partial result), and
// cuts them into G equal runs.  A run that falls on those units alone has no
// tile there.
constexpr int kSeqUnits = 1;

struct PlanState {
  int64_t T;       // units of all sequences
  int b0, x0, sb0;  // that sequence, its first flat tile, its first segment slot
  int ok;          // every sequence length was valid
};

__device__ __forceinline__ int nseg_of(int64_t x0, int64_t x1, int64_t T, int G) {
  return x1 > x0 ? group_of(x1 - 1, T, G) - group_of(x0, T, G) + 1 : 0;
}

// One warp builds the plan state of group g from the sequence lengths (two
// passes over them); with write_global it also writes the plan arrays the
// combine reads (the CTA holding group 0 does).
__device__ void plan_scan(const DecodeParams& p, int g, bool write_global, PlanState* ps) {
  const int lane = threadIdx.x & 31;
  int64_t T = 0;
  bool bad = false;
  for (int base = 0; base < p.B; base += 256) {  // pass 1: total tiles, validity (8 loads in flight)
    int L[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int b = base + u * 32 + lane;
      L[u] = b < p.B ? p.seqlens[b] : p.S;
    }
    int t = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (base + u * 32 + lane >= p.B) continue;
      if (L[u] < p.S || L[u] > p.Lmax) bad = true;
      else t += kSeqUnits + tiles_of(L[u]);
    }
    T += __reduce_add_sync(0xffffffffu, (unsigned)t);
  }
  bad = __any_sync(0xffffffffu, bad);
  const int64_t beg = (bad || T == 0) ? 0 : (int64_t)g * T / p.G;
  int64_t run_x = 0;
  int run_sb = 0, b0 = 0, x0 = 0, sb0 = 0;
  bool found = false;
  for (int base = 0; base < p.B && !bad && (write_global || !found); base += 32) {  // pass 2
    const int b = base + lane;
    const int t = b < p.B ? tiles_of(p.seqlens[b]) : 0;
    const int un = b < p.B ? kSeqUnits + t : 0;  // the sequence's units
    int it = un;  // inclusive scans over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, it, o);
      if (lane >= o) it += y;
    }
    const int64_t x = run_x + it - un;  // first unit of sequence b
    const int64_t xr = x + kSeqUnits;    // the unit of its first tile
    const int ns = nseg_of(xr, xr + t, T, p.G);
    int is = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) is += y;
    }
    const int sb = run_sb + is - ns;  // its first segment slot
    if (write_global && b < p.B) {
      p.prefix[b] = (int32_t)xr;
      p.gfirst[b] = t > 0 ? group_of(xr, T, p.G) : 0;
      p.segbase[b] = sb;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, t > 0 && x <= beg && beg < x + un);
    if (!found && hit) {
      const int src = __ffs(hit) - 1;
      b0 = __shfl_sync(0xffffffffu, b, src);
      x0 = __shfl_sync(0xffffffffu, (int)x, src);
      sb0 = __shfl_sync(0xffffffffu, sb, src);
      found = true;
    }
    run_x += __shfl_sync(0xffffffffu, it, 31);
    run_sb += __shfl_sync(0xffffffffu, is, 31);
  }
  if (lane == 0) {
    if (write_global) {
      p.prefix[p.B] = (int32_t)T;
      p.segbase[p.B] = run_sb;
      *p.plan_ok = bad ? 0u : 1u;
      if (bad) atomicOr(p.status, kDevErrBadSeqlen);
    }
    ps->T = T;
    ps->b0 = b0;
    ps->x0 = x0;
    ps->sb0 = sb0;
    ps->ok = (!bad && found) ? 1 : 0;
  }
}

// Tiles of group g in order, as a cursor that follows the sequences from the
// plan state on (prefix and segment slot carried along, lengths re-read).
struct TileCursor {
  int64_t beg, end, T;  // the group's units [beg, end) of T
  int64_t x0;           // first unit of sequence b
  int g, b, sb, t, tb, te, i, k, slot, L;
};

// Move c to the first sequence from c.b on that has tiles in the run.
__device__ __forceinline__ bool cursor_seq(const DecodeParams& p, TileCursor& c) {
  while (c.b < p.B && c.x0 < c.end) {
    const int L = p.seqlens[c.b];
    const int64_t xr = c.x0 + kSeqUnits, x1 = xr + tiles_of(L);
    if (x1 > c.beg && min(c.end, x1) > max(c.beg, xr)) {
      c.tb = (int)(max(c.beg, xr) - xr);
      c.te = (int)(min(c.end, x1) - xr);
      c.t = c.tb;
      c.slot = c.sb + (c.g - group_of(xr, c.T, p.G));
      c.L = L;
      return true;
    }
    c.sb += nseg_of(xr, x1, c.T, p.G);
    c.x0 = x1;
    ++c.b;
  }
  return false;
}

__device__ __forceinline__ bool cursor_start(const DecodeParams& p, int g, const PlanState& ps, TileCursor& c) {
  if (!ps.ok || ps.T <= 0) return false;
  c.T = ps.T;
  c.beg = (int64_t)g * ps.T / p.G;
  c.end = (int64_t)(g + 1) * ps.T / p.G;
  if (c.beg >= c.end) return false;
  c.g = g;
  c.i = 0;
  c.k = 0;
  c.b = ps.b0;
  c.x0 = ps.x0;
  c.sb = ps.sb0;
  return cursor_seq(p, c);
}

__device__ __forceinline__ bool cursor_next(const DecodeParams& p, TileCursor& c) {
  ++c.i;
  if (++c.t < c.te) return true;
  ++c.k;
  const int64_t xr = c.x0 + kSeqUnits, x1 = xr + tiles_of(c.L);
  c.sb += nseg_of(xr, x1, c.T, p.G);
  c.x0 = x1;
  ++c.b;
  return cursor_seq(p, c);
}

__device__ __forceinline__ TileInfo cursor_tile(const TileCursor& c) {
  return TileInfo{c.b, c.t, c.L, c.i, c.k, c.slot, min(c.L - c.t * kTok, kTok), c.t == c.tb, c.t == c.te - 1,
                  false};
}

// Visit every tile of group g in order (the plan state is in place).
template <class F>
__device__ __forceinline__ void for_each_tile(const DecodeParams& p, int g, const PlanState& ps, F&& f) {
  TileCursor c;
  for (bool have = cursor_start(p, g, ps, c); have; have = cursor_next(p, c))
    if (!f(cursor_tile(c))) return;
}

// The row warps' walk: optionally a dry visit of a stand-in tile first (no
// plan or global data needed, so it runs before the kernels this one depends
// on have finished), then the dependency wait, then every tile of group g.
// All visits go through the same call of f so that they run the same code.
template <class F>
__device__ __forceinline__ void for_each_tile_warm(const DecodeParams& p, int g, const PlanState& ps,
                                                   uint64_t* plan_bar, const WaitCtx& wc, F&& f) {
  TileInfo ti{0, 0, kTok, 0, 0, 0, kTok, true, false, true};
  TileCursor c;
  bool have = true;
  while (have) {
    if (!f(ti)) return;
    if (ti.dry) {
      pdl_wait();  // q_cat and the sequence lengths may come from the kernel before this one
      have = mbar_wait(plan_bar, 0, wc) && *wc.abort_flag == 0u && cursor_start(p, g, ps, c);
    } else {
      have = cursor_next(p, c);
    }
    if (have) ti = cursor_tile(c);
  }
}

// Score-CTA c-ring positions for tile i of segment k.  Every segment sends
// its 512 q~ columns through the c ring (two stages), every tile its cache
// rows (the same); stage h holds blocks 4h .. 4h + 3.  A segment's first
// tile interleaves them (q~ half 0, c half 0, q~ half 1, c half 1), so that
// its first QK^T half waits for two copies rather than three.  The k^R ring
// carries cache rows only (tile i at position i); q^R has its own buffer.
__device__ __forceinline__ int cpos_q(int i, int k, int h) { return kCPerTile * (i + k) + 2 * h; }
__device__ __forceinline__ int cpos_kv(int i, int k, int h, bool first) {
  return first ? kCPerTile * (i + k) + 2 * h + 1 : kCPerTile * (i + k + 1) + h;
}
constexpr int kBarC = 0, kBarR = kCStages;  // FULL / EMPTY sub-ranges of the two rings

// All 32 lanes wait; the outcome is made warp-uniform so that warp-collective
// tensor-memory instructions after it never run with a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// Exact 2^d for an integer d <= 0 (0 below the normal range).
__device__ __forceinline__ float exp2_int(int d) {
  return d <= -127 ? 0.f : __int_as_float((127 + d) << 23);
}

// Value CTA, end of a segment: the thread's half row of O (256 columns at
// tensor-memory address `ta`) leaves as 2^-e O / l in fp16, stored as
// [64 column octets][128 rows] of 16 bytes, so that each store of a warp
// covers 32 consecutive rows, 512 contiguous bytes (the epilogue is bound by
// an SM's store bandwidth, so halving the bytes against fp32 O halves its
// time).  O / l is a convex mix of cache rows; e >= 0 (stored beside, one per
// half row) is 0 unless some |O / l| reaches 2^15, and then the smallest
// power of two that brings every value of the half row below 2^15, so no
// cache value, however large, overflows fp16.  Kept out of line: it runs
// once per segment, and the per-tile loop around it stays small.
__device__ __noinline__ void store_partial(const DecodeParams& p, uint32_t ta, int hf, int r, int rb, int slot,
                                           float l_seg, bool valid) {
  const float inv0 = l_seg > 0.f ? 1.f / l_seg : 0.f;
  uint4* dst = p.opart + ((size_t)slot * p.n_rb + rb) * 64 * 128 + r;
  float amax = 0.f;
  int e = 0;
  for (int pass = 0; pass < 2; ++pass) {  // a second pass only when the first went out of range
    const float inv = inv0 * exp2_int(-e);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t v[64];
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
        tmem_ld32(ta + (uint32_t)(c * 64), lo);
        tmem_ld32(ta + (uint32_t)(c * 64 + 32), hi);
      }
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float* f = reinterpret_cast<const float*>(&v[8 * u]);
#pragma unroll
        for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(f[t]));
        dst[(size_t)(hf * 32 + c * 8 + u) * 128] =
            make_uint4(pack_f16x2_sat(f[0] * inv, f[1] * inv), pack_f16x2_sat(f[2] * inv, f[3] * inv),
                       pack_f16x2_sat(f[4] * inv, f[5] * inv), pack_f16x2_sat(f[6] * inv, f[7] * inv));
      }
    }
    const float top = amax * inv0;  // largest |O / l| of the half row
    if (pass == 1 || !(top >= 32768.f)) break;
    e = max(0, (int)((__float_as_uint(top) >> 23) & 0xFFu) - 141);  // top < 2^(biased exp - 126) <= 2^(15 + e)
  }
  if (valid) p.oexp[(((size_t)slot * p.n_rb + rb) * 128 + r) * 2 + hf] = (uint8_t)e;
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_c0, const __grid_constant__ CUtensorMap tm_kr,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                  const __grid_constant__ CUtensorMap tm_c1, const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int rb = cluster % p.n_rb, g = cluster / p.n_rb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SH = p.S * p.H;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    if (rank == 0) MLA_TRACE(p, TR_START, 0);
    *abort_flag = 0u;
    if (smem_u32(smem) & 1023u) {  // the swizzled tiles need 1 KB alignment
      *abort_flag = 1u;
      atomicOr(p.status, kDevErrInternal);
    }
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&bar[B_FULL + s], 1);
      mbar_init(&bar[B_EMPTY + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_SFULL + s], 1);
      mbar_init(&bar[B_SEMPTY + s], 256);
      mbar_init(&bar[B_PEMPTY + s], 1);
      mbar_init(&bar[B_PFULL + s], 1);
      mbar_init(&bar[B_PREADY + s], 256);
      mbar_init(&bar[B_PVDONE + s], 1);
    }
    for (int s = 0; s < 8; ++s) mbar_init(&bar[B_XCH + s], 64);
    mbar_init(&bar[B_XL], 256);
    mbar_init(&bar[B_OFREE], 256);
    mbar_init(&bar[B_DRAIN], 1);
    mbar_init(&bar[B_QRFULL], 1);
    mbar_init(&bar[B_QREMPTY], 1);
    // one arrival (the plan warp's); the stall test hook asks for two, so the
    // barrier never completes and every wait on it runs out
    mbar_init(&bar[B_PLAN], p.plan_arrivals);
    if (rank == 1) {  // first phase of each P slot expects one slot's bytes
      mbar_arrive_expect_tx(&bar[B_PFULL + 0], kPTx);
      mbar_arrive_expect_tx(&bar[B_PFULL + 1], kPTx);
    }
    fence_mbar_init_cluster();
    if (rank == 0) {
      tma_prefetch_desc(&tm_c0);
      tma_prefetch_desc(&tm_kr);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_qr);
    } else {
      tma_prefetch_desc(&tm_c1);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them remotely
  pdl_trigger();
  PlanState* plan = reinterpret_cast<PlanState*>(smem + kOffPlan);
  const bool rows = warp >= 4;
  if (warp == 3) {
    // The split plan, from the sequence lengths, which may come from the
    // kernels before this one like q_cat (row warps: after their dry visit).
    pdl_wait();
    plan_scan(p, g, blockIdx.x == 0, plan);
    __syncwarp();
    if (lane == 0 && rank == 0) MLA_TRACE(p, TR_PLAN, 0);
    if (lane == 0) mbar_arrive(&bar[B_PLAN]);
  } else if (!rows) {
    pdl_wait();
  }
  const uint32_t tmem = *tmem_slot;
  const bool run = rows || (warp < 3 && mbar_wait(&bar[B_PLAN], 0, wc) && plan->ok && *abort_flag == 0u);

  if (run && warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int qr_last = -1;  // last segment whose q^R was loaded
      int last_use[kRingSlots];
      for (int s = 0; s < kRingSlots; ++s) last_use[s] = -1;
      int cq = 0, rq = 0, q = 0;  // running positions: score c ring, score k^R ring, value ring
      // Issue one stage of a ring: wait for the slot, arm its barrier, copy.
      auto slot = [&](int base, int nst, int pos, uint32_t bytes) -> int {
        const int st = pos % nst;
        if (!mbar_wait(&bar[B_EMPTY + base + st], ((uint32_t)(pos / nst) & 1u) ^ 1u, wc)) return -1;
        mbar_arrive_expect_tx(&bar[B_FULL + base + st], bytes);
        last_use[base + st] = pos;
        return st;
      };
      for_each_tile(p, g, *plan, [&](const TileInfo& ti) {
        const int row0 = ti.b * p.Lmax + ti.t * kTok;
        if (rank == 0) {
          const int qrow0 = ti.b * SH + rb * 128;
          if (ti.first) {  // the segment's query rows: blocks 0..3 now, 4..7 after the tile's first c box
            const int st = slot(kBarC, kCStages, cq++, kCStage);
            if (st < 0) return false;
            tma_load_3d(smem + st * kCStage, &tm_q, &bar[B_FULL + kBarC + st], 0, qrow0, 0);
            if (!mbar_wait(&bar[B_QREMPTY], ((uint32_t)ti.k & 1u) ^ 1u, wc)) return false;
            mbar_arrive_expect_tx(&bar[B_QRFULL], kBlk0);
            qr_last = ti.k;
            tma_load_2d(smem + kOffQR, &tm_qr, &bar[B_QRFULL], 512, qrow0);
          }
          {  // the tile's k^R first: its MMAs open the tile's QK^T
            const int st = slot(kBarR, kRStages, rq++, kRStage);
            if (st < 0) return false;
            tma_load_2d(smem + kOffR + st * kRStage, &tm_kr, &bar[B_FULL + kBarR + st], 0, row0);
          }
          for (int h = 0; h < kCPerTile; ++h, ++cq) {
            if (ti.first && h == 1) {  // the query rows' second half, between the tile's two c boxes
              const int st = slot(kBarC, kCStages, cq++, kCStage);
              if (st < 0) return false;
              tma_load_3d(smem + st * kCStage, &tm_q, &bar[B_FULL + kBarC + st], 0, qrow0, 4);
            }
            const int st = slot(kBarC, kCStages, cq, kCStage);
            if (st < 0) return false;
            if (h == 0) MLA_TRACE(p, TR_TMA_ISSUE, ti.i);
            tma_load_3d(smem + st * kCStage, &tm_c0, &bar[B_FULL + kBarC + st], 0, row0, 4 * h);
          }
        } else {
          const int nsub = (ti.nvt + kSub - 1) / kSub;
          for (int u = 0; u < nsub; ++u, ++q) {  // 64-row stages of the 512 c columns
            const int st = slot(0, kStages1, q, kStage1);
            if (st < 0) return false;
            if (u == 0) MLA_TRACE(p, TR_V_TMA, ti.i);
            tma_load_3d(smem + st * kStage1, &tm_c1, &bar[B_FULL + st], 0, row0 + u * kSub, 0);
          }
        }
        return true;
      });
      // let every issued copy land before the CTA winds down
      for (int s = 0; s < kRingSlots; ++s) {
        if (last_use[s] < 0) continue;
        const int nst = rank == 0 ? (s < kBarR ? kCStages : kRStages) : kStages1;
        mbar_wait_drain(&bar[B_FULL + s], (uint32_t)(last_use[s] / nst) & 1u, wc);
      }
      if (qr_last >= 0) mbar_wait_drain(&bar[B_QRFULL], (uint32_t)qr_last & 1u, wc);
    }
  } else if (run && warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      if (rank == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, kTok, 0, 0);
        int ci = 0, ck = 0;  // the tile and segment whose q~ is being copied
        // Half h of the segment's q~ (its c-ring stage) into tensor memory.
        auto copy_q = [&](int h) -> bool {
          const int q = cpos_q(ci, ck, h), st = q % kCStages;
          if (!mbar_wait(&bar[B_FULL + kBarC + st], (uint32_t)(q / kCStages) & 1u, wc)) return false;
          tc_fence_after();
          const uint32_t sbase = smem_u32(smem + st * kCStage);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)  // 4 blocks x 4 slices of 16 columns
            tmem_cp_128x256b(tmem + kQCol + (uint32_t)(h * 16 + kk) * 8,
                             smem_desc(sbase + (kk >> 2) * kBlk0 + (kk & 3) * 32, 16, 1024, 2));
          mma_commit(&bar[B_EMPTY + kBarC + st]);  // the stage is free once the copy has read it
          return true;
        };
        for_each_tile(p, g, *plan, [&](const TileInfo& ti) {
          ci = ti.i;
          ck = ti.k;
          const int sb = ti.i & 1;                            // S buffer of this tile
          const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u;    // its phase
          if (ti.first) {
            // q~ of the segment: its two c stages go into tensor memory by
            // tcgen05.cp, after every MMA of the previous segment (which read
            // the old q~) has completed; a copy is ordered before this
            // thread's next MMAs.  Half 0 now, half 1 after the MMAs of the
            // tile's first c stage.  q^R must have landed in its buffer.
            if (ti.k > 0 && !mbar_wait(&bar[B_QREMPTY], (uint32_t)(ti.k - 1) & 1u, wc)) return false;
            if (!copy_q(0)) return false;
            if (!mbar_wait(&bar[B_QRFULL], (uint32_t)ti.k & 1u, wc)) return false;
          }
          if (!mbar_wait(&bar[B_SEMPTY + sb], sph ^ 1u, wc)) return false;
          const uint32_t d = tmem + (uint32_t)sb * 128u;
          {  // k^R against q^R, both 64 wide and K-major in shared memory; they open S
            const int q = ti.i, st = q % kRStages;
            if (!mbar_wait(&bar[B_FULL + kBarR + st], (uint32_t)(q / kRStages) & 1u, wc)) return false;
            tc_fence_after();
            MLA_TRACE(p, TR_QK_BEGIN, ti.i);
            const uint32_t sbase = smem_u32(smem + kOffR + st * kRStage), qbase = smem_u32(smem + kOffQR);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(d, smem_desc(qbase + kk * 32, 16, 1024, 2), smem_desc(sbase + kk * 32, 16, 1024, 2), idesc,
                     kk > 0 ? 1u : 0u);
            mma_commit(&bar[B_EMPTY + kBarR + st]);
          }
          for (int h = 0; h < kCPerTile; ++h) {  // c blocks 4h .. 4h + 3 against q~ from tensor memory
            // the second half of a new segment's q~ lands between the tile's c boxes;
            // its copy writes columns the first half's MMAs do not read
            if (ti.first && h == 1 && !copy_q(1)) return false;
            const int q = cpos_kv(ti.i, ti.k, h, ti.first), st = q % kCStages;
            if (!mbar_wait(&bar[B_FULL + kBarC + st], (uint32_t)(q / kCStages) & 1u, wc)) return false;
            if (h == kCPerTile - 1) MLA_TRACE(p, TR_QK_LAST, ti.i);
            tc_fence_after();
            const uint32_t sbase = smem_u32(smem + st * kCStage);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {  // 4 blocks x 4 K-steps of 16
              const int gk = h * 16 + kk;
              const uint64_t bd = smem_desc(sbase + (kk >> 2) * kBlk0 + (kk & 3) * 32, 16, 1024, 2);
              mma_ts(d, tmem + kQCol + (uint32_t)gk * 8, bd, idesc, 1u);
            }
            mma_commit(&bar[B_EMPTY + kBarC + st]);
          }
          if (ti.last) mma_commit(&bar[B_QREMPTY]);  // the next segment may replace q~ and q^R
          mma_commit(&bar[B_SFULL + sb]);
          MLA_TRACE(p, TR_QK_END, ti.i);
          return true;
        });
      } else {
        constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
        int q = 0;
        for_each_tile(p, g, *plan, [&](const TileInfo& ti) {
          const int slot = ti.i & 1;
          const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u;
          if (!mbar_wait(&bar[B_PREADY + slot], sph, wc)) return false;
          if (ti.first && ti.k > 0 && !mbar_wait(&bar[B_OFREE], (uint32_t)(ti.k - 1) & 1u, wc))
            return false;
          fence_proxy_async_cta();  // tail rows were zeroed through the generic proxy
          MLA_TRACE(p, TR_PV_BEGIN, ti.i);
          const int nk = (ti.nvt + 15) >> 4;  // K-steps of 16 tokens
          const uint32_t pbase = smem_u32(smem + kOffP + slot * kPSlot);
          for (int u = 0; u * kStepsPerSub < nk; ++u, ++q) {
            const int st = q % kStages1;
            if (!mbar_wait(&bar[B_FULL + st], (uint32_t)(q / kStages1) & 1u, wc)) return false;
            MLA_TRACE(p, TR_V_LAND, ti.i);
            tc_fence_after();
            const uint32_t sbase = smem_u32(smem + st * kStage1);
            for (int kt = 0; kt < kStepsPerSub && u * kStepsPerSub + kt < nk; ++kt) {
              const int gk = u * kStepsPerSub + kt;
              const uint64_t ad = smem_desc(pbase + (gk >> 2) * 16384 + (gk & 3) * 32, 16, 1024, 2);
#pragma unroll
              for (int n = 0; n < 2; ++n) {  // N = 512 latent columns as 2 x 256
                const uint64_t bd = smem_desc(sbase + n * 4 * kBlk1 + kt * 2048, kBlk1, 1024, 2);
                mma_ss(tmem + (uint32_t)n * 256, ad, bd, idesc, (gk > 0 || !ti.first) ? 1u : 0u);
              }
            }
            mma_commit(&bar[B_EMPTY + st]);
          }
          mma_commit(&bar[B_PVDONE + slot]);
          MLA_TRACE(p, TR_PV_END, ti.i);
          return true;
        });
      }
      mma_commit(&bar[B_DRAIN]);  // every MMA has finished before tensor memory is released
      mbar_wait_drain(&bar[B_DRAIN], 0, wc);
    }
  } else if (run && warp == 2 && rank == 1) {
    if (lane == 0) {
      // -------------------------------------------- value CTA: P-slot releaser
      for_each_tile(p, g, *plan, [&](const TileInfo& ti) {
        const int slot = ti.i & 1;
        if (!mbar_wait(&bar[B_PVDONE + slot], (uint32_t)(ti.i >> 1) & 1u, wc)) return false;
        MLA_TRACE(p, TR_PV_DONE, ti.i);
        mbar_arrive_remote(&bar[B_PEMPTY + slot], 0);
        return true;
      });
    }
  } else if (run && warp >= 4) {
    // ------------------------------------------------ warps 4..11: two threads per row
    const int q4 = warp & 3;          // tensor-memory lane quadrant of this warp
    const int hf = (warp - 4) >> 2;   // half of the row's columns this thread owns
    const int r = q4 * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const int gr = rb * 128 + r;
    const bool valid = gr < SH;
    const int s_r = valid ? gr / p.H : 0;

    if (rank == 0) {
      // ---------------------------------------- scores + online softmax
      float* xch = reinterpret_cast<float*>(smem + kOffXch);                  // [2][2][128]
      float* xl = reinterpret_cast<float*>(smem + kOffXch + 2 * 2 * 128 * 4);  // [128]
      // P, the rescale exponent and the row sum go straight into the value
      // CTA's P slot as asynchronous remote stores, each counted (in bytes) on
      // that slot's barrier there.
      const uint32_t p_remote = map_to_cta(smem_u32(smem + kOffP), 1);
      const uint32_t pfull_remote = map_to_cta(smem_u32(&bar[B_PFULL]), 1);
      float m_ref = -INFINITY, l = 0.f;
      int limit = 0;
      for_each_tile_warm(p, g, *plan, &bar[B_PLAN], wc, [&](const TileInfo& ti) {
        if (ti.first) {
          limit = valid ? ti.L - p.S + s_r + 1 : 0;
          m_ref = -INFINITY;
          l = 0.f;
        }
        const int slot = ti.i & 1;  // S buffer, exchange slot and P slot of this tile
        const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u;
        if (!ti.dry && !warp_wait(&bar[B_SFULL + slot], sph, wc)) return false;
        if (!ti.dry && threadIdx.x == 128) MLA_TRACE(p, TR_S_READY, ti.i);
        tc_fence_after();
        const uint32_t sc = tl + (uint32_t)(slot * 128 + hf * 64);  // this thread's 64 score columns
        const int nv = min(max(limit - ti.t * kTok - hf * 64, 0), 64);

        // The scores are read from tensor memory twice, 16 at a time, in
        // rolled loops: the code stays small (the instruction stream of the
        // row warps competes with the other roles' for the SM's instruction
        // caches), and the other S buffer lets the next tile's QK^T run
        // meanwhile.
        float mx = -INFINITY;  // max of the raw scores; the scale is positive
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(sc + (uint32_t)(c * 16), v);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (c * 16 + u < nv) mx = fmaxf(mx, __uint_as_float(v[u]));
        }
        mx *= p.scale_log2;
        if (!ti.dry && threadIdx.x == 128) MLA_TRACE(p, TR_SM_MAX, ti.i);
        // Both threads of the row (same quadrant, warps q4 and q4 + 4) need the
        // same new reference exponent, which depends on the row maximum only
        // through ceil(max): for an integer m, max > m + 8 iff ceil(max) > m + 8.
        // So the two halves exchange ceil(max) (-inf when no column is visible).
        const float cm = ceilf(mx);
        xch[(slot * 2 + hf) * 128 + r] = cm;
        if (!ti.dry) {
          mbar_arrive(&bar[B_XCH + slot * 4 + q4]);
          if (!warp_wait(&bar[B_XCH + slot * 4 + q4], sph, wc)) return false;
        }
        if (!ti.dry && threadIdx.x == 128) MLA_TRACE(p, TR_SM_XCH, ti.i);
        const float cmax = fmaxf(cm, xch[(slot * 2 + (hf ^ 1)) * 128 + r]);
        int ex = 0;  // rescale 2^-ex of O and l; 255 stands for 0
        if (cmax > m_ref + 8.f) {  // never for -inf; m is a float holding an integer
          ex = (m_ref == -INFINITY) ? 255 : (int)fminf(cmax - m_ref, 255.f);
          l = (ex == 255) ? 0.f : l * exp2_int(-ex);
          m_ref = cmax;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;

        // the value CTA's P slot is free once its P . C of two tiles ago completed
        if (!ti.dry && !warp_wait(&bar[B_PEMPTY + slot], sph ^ 1u, wc)) return false;
        if (!ti.dry && threadIdx.x == 128) MLA_TRACE(p, TR_SM_SLOT, ti.i);
        const uint32_t pslot = p_remote + (uint32_t)(slot * kPSlot), pbar = pfull_remote + (uint32_t)slot * 8;
        const uint32_t prow = pslot + (uint32_t)(hf * 16384 + r * 128);
        float lsum0 = 0.f, lsum1 = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {  // 2^(s scale log2 e - m), 16 columns per pass
          uint32_t v[16];
          tmem_ld16(sc + (uint32_t)(c * 16), v);
          tmem_wait_ld();
          uint32_t pk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int col = c * 16 + 2 * u;
            const float e0 = col < nv ? ex2_approx(fmaf(__uint_as_float(v[2 * u]), p.scale_log2, -mu)) : 0.f;
            const float e1 =
                col + 1 < nv ? ex2_approx(fmaf(__uint_as_float(v[2 * u + 1]), p.scale_log2, -mu)) : 0.f;
            pk[u] = pack_bf16x2(e0, e1);
            const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[u]);
            lsum0 += __low2float(b2);
            lsum1 += __high2float(b2);
          }
          // 128-byte swizzle: chunk ch of row r sits at ch ^ (r & 7)
          if (!ti.dry) {
            st_async_v4(prow + (uint32_t)(((2 * c) ^ (r & 7)) << 4), pk[0], pk[1], pk[2], pk[3], pbar);
            st_async_v4(prow + (uint32_t)(((2 * c + 1) ^ (r & 7)) << 4), pk[4], pk[5], pk[6], pk[7], pbar);
          }
        }
        tc_fence_before();
        if (!ti.dry) mbar_arrive(&bar[B_SEMPTY + slot]);  // this S buffer has been read
        if (!ti.dry && threadIdx.x == 128) MLA_TRACE(p, TR_P_SENT, ti.i);
        l += lsum0 + lsum1;
        float l_seg = 0.f;  // segment end: the row's whole sum (both halves), for hf = 0
        if (ti.last && !ti.dry) {
          if (hf == 1) xl[r] = l;
          mbar_arrive(&bar[B_XL]);
          if (!warp_wait(&bar[B_XL], (uint32_t)ti.k & 1u, wc)) return false;
          l_seg = l + xl[r];
          // the next segment's exchange reuses xl only after its own tiles'
          // row-max exchanges, which both threads pass after reading it here
        }
        if (ti.dry) return true;
        if (hf == 0) {  // the value CTA rescales O with ex and normalises it with l at a segment end
          st_async_b32(pslot + (uint32_t)(kOffPEx + r * 4), (uint32_t)ex, pbar);
          st_async_b32(pslot + (uint32_t)(kOffPL + r * 4), __float_as_uint(l_seg), pbar);
        }
        if (ti.last && hf == 0 && valid)  // segment end: (m, l) of the row
          p.ml[((size_t)ti.slot * p.n_rb + rb) * 128 + r] = make_float2(mu, l_seg);
        return true;
      });
    } else {
      // ---------------------------------------- rescale, tail zeroing, epilogue
      const int wt = threadIdx.x - 128;  // 0..255
      int q = 0;  // running stage counter (as the producer's)
      for_each_tile_warm(p, g, *plan, &bar[B_PLAN], wc, [&](const TileInfo& ti) {
        const int slot = ti.i & 1;
        const uint32_t sph = (uint32_t)(ti.i >> 1) & 1u;
        const int nsub = (ti.nvt + kSub - 1) / kSub;
        const int q0 = q;
        if (!ti.dry) q += nsub;
        if (!ti.dry && !warp_wait(&bar[B_PFULL + slot], sph, wc)) return false;
        if (!ti.dry && wt == 0) MLA_TRACE(p, TR_P_FULL, ti.i);
        const int ex = (int)reinterpret_cast<const volatile uint32_t*>(smem + kOffP + slot * kPSlot + kOffPEx)[r];
        const float l_seg = ti.last
            ? reinterpret_cast<const volatile float*>(smem + kOffP + slot * kPSlot + kOffPL)[r] : 0.f;
        const float alpha = ex == 255 ? 0.f : exp2_int(-ex);
        if (!ti.dry && wt == 0) mbar_arrive_expect_tx(&bar[B_PFULL + slot], kPTx);  // arm the slot's next phase
        const bool need = !ti.first && alpha != 1.f;
        if (__any_sync(0xffffffffu, need)) {
          // O rows change only after the previous tile's P . C has completed
          if (!warp_wait(&bar[B_PVDONE + (slot ^ 1)], (uint32_t)((ti.i - 1) >> 1) & 1u, wc)) return false;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t v[32];
            const uint32_t a = tl + (uint32_t)(hf * 256 + c * 32);
            tmem_ld32(a, v);
            tmem_wait_ld();
            if (need) {
#pragma unroll
              for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * alpha);
            }
            tmem_st32(a, v);
          }
          tmem_wait_st();
        }
        if (ti.dry) return true;
        if (ti.nvt & 15) {
          // cache rows past the sequence end inside the last 16-row MMA step hold
          // arbitrary bytes; their weights are 0 but 0 * NaN is not, so zero them
          const int u = ti.nvt / kSub, qs = q0 + u, st = qs % kStages1;
          if (!warp_wait(&bar[B_FULL + st], (uint32_t)(qs / kStages1) & 1u, wc)) return false;
          const int z0 = ti.nvt - u * kSub, nzr = ((ti.nvt + 15) & ~15) - ti.nvt;
          uint8_t* sb = smem + st * kStage1;
          for (int idx = wt; idx < nzr * 64; idx += 256) {
            const int blk = idx / (nzr * 8), rem = idx - blk * (nzr * 8);
            *reinterpret_cast<uint4*>(sb + blk * kBlk1 + (z0 + (rem >> 3)) * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_cta();
        }
        tc_fence_before();
        mbar_arrive(&bar[B_PREADY + slot]);
        if (ti.last) {
          if (!warp_wait(&bar[B_PVDONE + slot], sph, wc)) return false;
          if (wt == 0) MLA_TRACE(p, TR_EPI_BEGIN, ti.k);
          tc_fence_after();
          store_partial(p, tl + (uint32_t)(hf * 256), hf, r, rb, ti.slot, l_seg, valid);
          tc_fence_before();
          if (wt == 0) MLA_TRACE(p, TR_EPI_END, ti.k);
          mbar_arrive(&bar[B_OFREE]);
        }
        return true;
      });
    }
  }

  // ------------------------------------------------ wind down
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) MLA_TRACE(p, TR_END, rank);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  cluster_sync();
}

}  // namespace mla
