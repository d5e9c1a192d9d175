// Tiled FlashAttention forward for sm_103a: dense, causal, ragged (per-batch
// lengths), GQA and block-sparse (compact KV-block lists), D = Dv in {64, 128}.
//
// One CTA owns up to two 128-row query tiles ("slots") that are processed in
// ping-pong so that the softmax of one overlaps the tensor-core work of the
// other.  Work split inside the CTA (512 threads, four warpgroups):
//   warps 0-3   softmax of slot 0 (one thread per query row), including the
//               correction O *= exp2(m_old - m_new) of its rows when the max
//               moves, then the slot's epilogue (O / l, LSE)
//   warps 4-7   softmax and epilogue of slot 1
//   warps 8-11  V converter during the tile loop (bf16 V)
//   warp  12    TMA producer: Q tiles, then K / V tiles into a ring of stages
//   warp  13    TMEM allocator and tcgen05.mma issuer
//   warp  14    MMA scheduler: waits on the mbarriers of the next MMA groups and
//               releases them to warp 13 through named barriers
//   warp  15    L2 prefetch of the first tiles, outside the setup barrier
// Q and K are bf16 or fp16; the P.V product reads fp16 V (P and V share the
// fp16 type): a bf16 V is converted in shared memory by warps 8-11 as its tiles
// arrive (kConvV), or was converted beforehand by the caller.
// The softmax warpgroups raise their register budget with setmaxnreg; the
// other two lower theirs.
//
// TMEM (512 columns): S_t / P_t of slot t at column 128 t, O_t at 256 + 128 t.
// P is written over S as fp16 (64 columns); rows that see few keys also get a
// second fp16 term P_lo = p - fp16(p) in columns 64..127 (hi + lo split).
//
// The online softmax follows the loop invariant of the FlashAttention
// correctness-verification page (ai6s.net), section "Formal verification
// outline": per row a running max m and sum l, O rescaled by exp(m_old - m_new)
// when the max moves.  The move is gated by the lazy-rescale rule of the
// sparse-MLA page (cf-1.com), section "Verifying the threshold branch from
// source": keep the stale max while the block max exceeds it by no more than
// `threshold` log2 units (0 = exact running max).
#pragma once
#include <type_traits>

#include "fa_ptx.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per KV tile
constexpr int kTiledThreads = 512;
// setmaxnreg budgets per warpgroup (two softmax, correction, producer/MMA/converter);
// their sum over the four warpgroups must not exceed 4 x the launch budget of
// 128 registers per thread (the host checks the compiled count before launch)
constexpr int kSoftmaxRegs = 200;
constexpr int kCorrRegs = 56;
constexpr int kOtherRegs = 56;
constexpr int kRegsNeeded = (2 * kSoftmaxRegs + kCorrRegs + kOtherRegs + 3) / 4;
static_assert(kSoftmaxRegs % 8 == 0 && kCorrRegs % 8 == 0 && kOtherRegs % 8 == 0,
              "setmaxnreg takes multiples of 8");
static_assert(kRegsNeeded <= 65536 / kTiledThreads, "register split exceeds the register file");
constexpr int kMaxSel = 512;      // longest block list a CTA stages in smem
constexpr int kHiLoKeys = 256;    // rows with fewer valid keys use the hi+lo P split
constexpr int kMaxSplit = 8;      // most pieces a unit's KV tiles are split into
// hardware named barriers (0 is __syncthreads, the teardown): 1-2 scheduler ->
// issuer release of groups 0 and 1, 3-4 issuer -> scheduler "group issued", 5-6
// "P ready" of slot t (its softmax warps and the scheduler -> issuer: P written
// and the group's copies landed), 7-8 the epilogue of slot t (its softmax
// warps), 9 the setup (warp 15 only arrives)
constexpr int kBarPReady = 5;
constexpr int kBarEpi = 7;
constexpr int kBarSetup = 9;
constexpr int kPReadyCount = kBM + 64;   // slot's softmax threads, scheduler, issuer

enum : int { kStatusTimeout = 1, kStatusRange = 2 };

struct TiledParams {
  CUtensorMap tm_q, tm_k, tm_v;
  void* o;
  void* o_lo;       // optional: o's rounding residual, same type and layout (or null)
  float* lse;
  const int* seqlens;
  const int* blk_idx;
  long long blk_stride_b, blk_stride_h;
  int max_sel;
  int B, Hq, Hkv, Sq, Skv;
  int G;            // Hq / Hkv
  int mask;         // 0 none, 1 causal, 2 causal inside the diagonal block
  int pair_mode;    // 0: slots = query tiles 2p, 2p+1 of one head; 1: heads 2p, 2p+1 at one tile
  int n_qt;         // ceil(Sq / 128)
  int units_per_q;  // units that share one query position
  int n_qpos;       // query positions (tile pairs or tiles)
  int head_major;   // 1: units ordered by (batch, head) first (block lists)
  int kv_split;     // pieces per unit along the KV tiles (1: no split); dense only
  float* part_o;    // kv_split > 1: O / l of every piece, fp32 [kv_split][B*Hq*Sq][Dv]
  float* part_lse;  // kv_split > 1: LSE of every piece (-inf: no key) [kv_split][B*Hq*Sq]
  float scale, scale_log2, threshold;
  long long timeout_ns;
  int* status;
  unsigned long long* trace;   // cycle-stamped events of the first CTAs (trace builds only)
  // The operator doc's optional terms (kExtras launches only):
  int win_mode;                // 0: none; 1: keys i - pre_tokens <= j <= i + next_tokens;
                               // 2: bottom-right causal, j <= i + kv_len - q_len
  int pre_tokens, next_tokens; // win_mode 1 (clamped by the host to +-(Sq + Skv))
  const uint8_t* amask;        // explicit mask or null: nonzero byte = key masked
  long long am_sb, am_sh, am_sq;   // its strides (elements) over batch, head, query row
  int alibi;                   // score bias -slope_h |i - j| (1) or -slope_h sqrt|i - j| (2),
                               // slope_h = 2^(-8 (h + 1) / Hq)
  const uint16_t* pse;         // bias tensor or null: q's type, strides below (elements)
  long long pse_sb, pse_sh, pse_sq;
  int pse_type;                // 0: s * scale + pse; 1: (s + pse) * scale
  // dropout, O = (P * M / keep_prob) V: element (b, h, i, j) of the
  // row-major [B, Hq, Sq, Skv] grid is kept when byte (index % 16) of the
  // Philox4x32-10 output for counter drop_ctr0 + index / 16 is below keep_thr
  int keep_thr;                // 256: no dropout
  float keep_prob;
  uint32_t drop_key0, drop_key1;
  unsigned long long drop_ctr0;
  // FP8 inputs (q, k and v hold the exact fp16 values of x_q): per-block
  // dequant scales [planes][blocks of 128 rows] (null: none).  S of a (query
  // tile, key tile) pair is scaled by d_q d_k; P of a key tile by d_v / dmax,
  // dmax the largest d_v of the slot's tiles (so the fp16 P operand neither
  // overflows nor falls into subnormals for the tiles that matter), and dmax
  // joins 1 / l in the epilogue
  const float* dsq;
  const float* dsk;
  const float* dsv;
  int ds_nbq, ds_nbk;
};

// Trace points: compiled only with -DFA_TRACE (a profiling build); otherwise
// they expand to nothing.  Every tracing thread owns one region of the buffer
// (no atomics): region = CTA * kTraceRoles + role, slot 0 of a region holds
// its count.  Each record is clock64 << 24 | tag << 16 | slot << 15 | j.
constexpr int kTraceCtas = 8;
constexpr int kTraceRoles = 8;
constexpr int kTraceCap = 1024;
#ifdef FA_TRACE
__device__ __forceinline__ void fa_trace(const TiledParams& p, int role, int& n, int tag, int t,
                                         int j) {
  if (p.trace == nullptr || blockIdx.x >= kTraceCtas) return;
  unsigned long long* buf = p.trace + ((size_t)blockIdx.x * kTraceRoles + role) * kTraceCap;
  ++n;
  if (n < kTraceCap)
    buf[n] = ((unsigned long long)clock64() << 24) | ((unsigned long long)tag << 16) |
             ((unsigned long long)(t & 1) << 15) | (unsigned long long)(j & 0x7FFF);
  buf[0] = (unsigned long long)n;
}
#define FA_TR_ROLE(r) \
  int tr_n = 0;       \
  const int tr_role = (r)
#define FA_TR(tag, t, j) fa_trace(p, tr_role, tr_n, tag, t, j)
#else
#define FA_TR_ROLE(r) ((void)0)
#define FA_TR(tag, t, j) ((void)0)
#endif
// tags: 1 S ready (softmax), 2 P written (softmax), 5 stage load issued
// (producer), 6 QK issued, 7 PV issued, 9 dependencies met (MMA), 10 epilogue
// start, 11 epilogue end, 12 kernel start, 13 kernel end

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <int D, int NS>
struct TiledSmem {
  static constexpr int kQBytes = kBM * D * 2;           // one query tile
  static constexpr int kStageBytes = kBN * D * 2;       // one K or V tile (Dv == D)
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = 2 * kQBytes;
  static constexpr int kListOff = kStageOff + NS * kStageBytes;
  static constexpr int kBarOff = kListOff + 2 * kMaxSel * 4;
  // barriers: q_full[2], full[NS], empty[NS], s_full[2], o_ready[2], drain,
  // ready[NS] (a load passed the V converter)
  static constexpr int kNumBars = 2 + 2 * NS + 4 + 1 + NS;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag, slot info
  static constexpr int kBytes = kMiscOff + 64;
  static constexpr int kAlloc = kBytes + 1024;              // slack for 1024-byte alignment
};

struct WaitCtx {
  volatile int* abort;
  int* status;
  long long timeout;
};

// Bounded wait on an mbarrier phase.  Returns false (and stops every other
// wait of the CTA) once the limit passes or another thread gave up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, WaitCtx c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    // suspended in hardware until the phase completes (or ~20 us pass)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*c.abort) return false;
    if ((long long)(globaltimer_ns() - t0) > c.timeout) {
      *c.abort = 1;
      atomicOr(c.status, kStatusTimeout);
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag (teardown: let copies and MMAs in
// flight finish before their shared memory or TMEM is released).  It waits at
// least kDrainNs, whatever the caller's wait limit, since a short limit must
// not cut a copy's landing short.
constexpr long long kDrainNs = 100000000;   // 100 ms
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, long long timeout) {
  if (timeout < kDrainNs) timeout = kDrainNs;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > timeout) return;
  }
}

// KV tiles of a dense (not block-sparse) query tile: up to the causal bound
// and the batch's length; 0 for a tile past the query length.
__device__ __forceinline__ int dense_tiles(int qt, int n_qt, int q_len, int kv_len, int mask) {
  const int q0 = qt * kBM;
  if (qt >= n_qt || q0 >= q_len || kv_len <= 0) return 0;
  int nkv = (kv_len + kBN - 1) / kBN;
  if (mask == 1) nkv = min(nkv, min(q0 + kBM - 1, q_len - 1) / kBN + 1);
  return nkv;
}

// One piece of a unit split along its KV tiles: the slots' ranges [0, n0) and
// [0, n1) are cut at the same tile boundaries, every ceil(max(n0, n1) /
// kv_split) tiles; a slot's piece is [lo, min(n, hi)), possibly empty.
// (Unsplit launches skip the division: the setup is on every CTA's serial path.)
struct Piece {
  int lo, hi;
};
__device__ __forceinline__ Piece piece_range(int n0, int n1, int piece, int kv_split) {
  const int nmax = n0 > n1 ? n0 : n1;
  if (kv_split == 1) return Piece{0, nmax};
  const int chunk = (nmax + kv_split - 1) / kv_split;
  const int lo = min(piece * chunk, nmax);
  return Piece{lo, min(lo + chunk, nmax)};
}
__device__ __forceinline__ int piece_count(int n, Piece pc) { return max(0, min(n, pc.hi) - pc.lo); }

// The unit a launch index stands for.  Units are numbered heaviest query
// position first (u / units_per_q from the last position).  Block lists give
// every query block its own list, typically of one length, so that order buys
// no balance there; they run one head's positions after another instead, so
// that the CTAs in flight share a few heads' K and V in L2.
__device__ __forceinline__ int unit_of(const TiledParams& p, int idx) {
  if (!p.head_major) return idx;
  const int bh = idx / p.n_qpos, qpos = idx - bh * p.n_qpos;
  return (p.n_qpos - 1 - qpos) * p.units_per_q + bh;
}

// Number of SMs of this GPU.
__device__ __forceinline__ uint32_t sm_count() {
  uint32_t n;
  asm("mov.u32 %0, %%nsmid;" : "=r"(n));
  return n;
}

// L2 prefetch of a unit's first tiles (its query tiles, the first two K and V
// tiles of a dense unit), computed from the kernel's arguments alone.
template <int D, bool kSplit>
__device__ __noinline__ void prefetch_unit_l2(const TiledParams& p) {
  constexpr int kBoxes = D / 64;
  const int kv_split = kSplit ? p.kv_split : 1;
  const int u = unit_of(p, kSplit ? (int)blockIdx.x / kv_split : (int)blockIdx.x);
  const int piece = kSplit ? (int)(blockIdx.x % (unsigned)kv_split) : 0;
  const int qpos = p.n_qpos - 1 - u / p.units_per_q;
  const int bh = u % p.units_per_q;
  int b, h0, h1, qt0, qt1;
  if (p.pair_mode == 0) {
    b = bh / p.Hq;
    h0 = h1 = bh % p.Hq;
    qt0 = 2 * qpos;
    qt1 = 2 * qpos + 1;
  } else {
    const int hpairs = p.Hq / 2;
    b = bh / hpairs;
    h0 = 2 * (bh % hpairs);
    h1 = h0 + 1;
    qt0 = qt1 = qpos;
  }
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  for (int t = 0; t < 2; ++t) {
    const int qt = t ? qt1 : qt0;
    if (qt >= p.n_qt) continue;
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_prefetch_l2_3d(&p.tm_q, 64 * bx, qt * kBM, b * p.Hq + (t ? h1 : h0));
  }
  if (p.blk_idx == nullptr && p.win_mode != 1) {
    // (a key window starts elsewhere) the per-batch lengths are read only
    // after the wait: a prefetched tile that turns out unused costs only
    // bandwidth
    const int f0 = dense_tiles(qt0, p.n_qt, p.Sq, p.Skv, p.mask);
    const int f1 = dense_tiles(qt1, p.n_qt, p.Sq, p.Skv, p.mask);
    const Piece pc = piece_range(f0, f1, piece, kv_split);
    const int nf = min(2, pc.hi - pc.lo);
    const int kvh = h0 / p.G;
    for (int j = 0; j < nf; ++j)
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_prefetch_l2_3d(&p.tm_k, 64 * bx, (pc.lo + j) * kBN, b * p.Hkv + kvh);
        tma_prefetch_l2_3d(&p.tm_v, 64 * bx, (pc.lo + j) * kBN, b * p.Hkv + kvh);
      }
  }
}

// Keys visible from query row i under the optional terms, before the explicit
// mask: [ext_key_lo(i), ext_key_hi(i)] (empty when hi < lo; hi = -1 for a row
// past the batch's length).
__device__ __forceinline__ int ext_key_lo(const TiledParams& p, int i) {
  return p.win_mode == 1 ? max(0, i - p.pre_tokens) : 0;
}
__device__ __forceinline__ int ext_key_hi(const TiledParams& p, int i, int q_len, int kv_len) {
  if (i >= q_len) return -1;
  int hi = kv_len - 1;
  if (p.mask == 1) hi = min(hi, i);                       // top-left causal
  if (p.win_mode == 1) hi = min(hi, i + p.next_tokens);
  if (p.win_mode == 2) hi = min(hi, i + kv_len - q_len);  // bottom-right causal
  return hi;
}

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): per round (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^
// k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)), the key advanced by the Weyl
// increments between rounds; the dropout generator of the FlashAttentionScore-
// Grad write-up, section 5.3.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The order in which the MMA warp consumes K / V tiles, as a numbered event
// list: 0 = QK(0,0), 1 = QK(1,0), then per iteration j four events PV(0,j),
// QK(0,j+1), PV(1,j), QK(1,j+1).  `load` marks the first use of a tile (a
// new ring stage), `rel` the last.  With `shared`, slot 1 reads the tiles slot
// 0 loaded (same KV head and KV tile sequence, n0 <= n1).
struct Event {
  bool valid, pv, load, rel;
  int t, j;
};
__device__ __forceinline__ int num_events(int n0, int n1) {
  const int n = n0 > n1 ? n0 : n1;
  return n > 0 ? 2 + 4 * n : 0;
}
__device__ __forceinline__ Event event_at(int e, int n0, int n1, bool shared) {
  Event ev;
  if (e < 2) {
    ev.pv = false;
    ev.t = e;
    ev.j = 0;
  } else {
    const int r = (e - 2) & 3;
    const int j = (e - 2) >> 2;
    ev.pv = (r & 1) == 0;
    ev.t = r >> 1;
    ev.j = ev.pv ? j : j + 1;
  }
  const int nt = ev.t ? n1 : n0;
  ev.valid = ev.j < nt;
  ev.load = shared ? (ev.t == 0 || ev.j >= n0) : true;
  ev.rel = shared ? (ev.t == 1) : true;
  return ev;
}

// kConvV: V arrives as bf16 and the epilogue warpgroup, idle during the tile
// loop, converts each V tile to fp16 in shared memory before the MMA reads it.
// kSplit: the launch cuts units into KV pieces (p.kv_split > 1); an unsplit
// launch compiles without the piece bookkeeping, which costs ~1-2 % of the
// loop's time even when every unit is one piece.
// kExtras: the operator doc's optional terms (p.win_mode, p.amask, p.alibi);
// each slot walks its own list of KV tiles (its window), scores are scaled to
// log2 units before the mask and the row max.
template <int D, bool kBF16, int NS, bool kConvV, bool kSplit, bool kExtras = false>
__global__ void __launch_bounds__(kTiledThreads, 1)
    fa_fwd_tiled_kernel(const __grid_constant__ TiledParams p) {
  using SM = TiledSmem<D, NS>;
  constexpr int Dv = D;
  constexpr int kKSteps = D / 16;     // QK^T k-steps of 16
  constexpr int kBoxes = D / 64;      // 128-byte swizzle boxes per row
  constexpr uint32_t kIdescQK = idesc_f16(kBM, kBN, kBF16, false);
  constexpr uint32_t kIdescPV = idesc_f16(kBM, Dv, false, true);   // fp16 P, fp16 V (MN-major)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + SM::kQOff;
  const uint32_t sStage = sbase + SM::kStageOff;
  int* s_list = reinterpret_cast<int*>(smem + SM::kListOff);
  const uint32_t bar0 = sbase + SM::kBarOff;
  auto BAR_QFULL = [=](int t) { return bar0 + 8u * t; };
  auto BAR_FULL = [=](int s) { return bar0 + 8u * (2 + s); };
  auto BAR_EMPTY = [=](int s) { return bar0 + 8u * (2 + NS + s); };
  auto BAR_SFULL = [=](int t) { return bar0 + 8u * (2 + 2 * NS + t); };
  auto BAR_OREADY = [=](int t) { return bar0 + 8u * (4 + 2 * NS + t); };
  const uint32_t BAR_DRAIN = bar0 + 8u * (6 + 2 * NS);
  // with kConvV every ring load passes the converter (V tiles converted, K
  // tiles untouched) and the MMA side waits here instead of on BAR_FULL
  auto BAR_READY = [=](int s) { return kConvV ? bar0 + 8u * (7 + 2 * NS + s) : bar0 + 8u * (2 + s); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SM::kMiscOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + SM::kMiscOff + 4);
  int* s_slot = reinterpret_cast<int*>(smem + SM::kMiscOff + 8);   // [2] n, [2] hilo

  // The next call on the stream may be scheduled once every CTA of this one
  // has started (its CTAs then wait here for this grid to finish); nothing
  // below touches global memory before the previous kernel has completed.
  pdl_launch_dependents();
  // While the previous kernel on the stream may still run, warp 15 warms L2
  // with the first tiles of this CTA's unit (a prefetch only reads into the
  // cache, which stays coherent with that kernel's later writes): the first
  // wave of CTAs is scheduled during the previous kernel's tail, and its first
  // loads then come from L2 instead of every CTA reading HBM at once.  Later
  // CTAs start after that kernel has finished and load at once instead.  The
  // warp has no other role and arrives at the setup barrier first: the
  // prefetch's code is fetched cold at a launch with nothing before it, and
  // the setup must not wait for it (3-4 us per launch on the dense benchmark).
  if (threadIdx.x >= 32 * 15) {
    named_arrive(kBarSetup, kTiledThreads);
    if (threadIdx.x == 32 * 15 && blockIdx.x < sm_count()) prefetch_unit_l2<D, kSplit>(p);
    __syncwarp();
    regs_dec<kOtherRegs>();   // with the other warps of the fourth warpgroup
    __syncthreads();          // the teardown
    return;
  }
  pdl_wait_prior();

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---------------------------------------------------------------- unit
  const int kv_split = kSplit ? p.kv_split : 1;
  // pieces of one unit are neighbours
  const int u = unit_of(p, kSplit ? (int)blockIdx.x / kv_split : (int)blockIdx.x);
  const int piece = kSplit ? (int)(blockIdx.x % (unsigned)kv_split) : 0;
  const int qpos = p.n_qpos - 1 - u / p.units_per_q;   // heaviest query positions first
  const int bh = u % p.units_per_q;
  int b, h0, h1, qt0, qt1;
  if (p.pair_mode == 0) {
    b = bh / p.Hq;
    h0 = h1 = bh % p.Hq;
    qt0 = 2 * qpos;
    qt1 = 2 * qpos + 1;
  } else {
    const int hpairs = p.Hq / 2;
    b = bh / hpairs;
    h0 = 2 * (bh % hpairs);
    h1 = h0 + 1;
    qt0 = qt1 = qpos;
  }
  const int kvh = h0 / p.G;   // both slots share it (GQA pairs never straddle a group)
  const int q_len = p.seqlens ? min(p.seqlens[b], p.Sq) : p.Sq;
  const int kv_len = p.seqlens ? min(p.seqlens[b], p.Skv) : p.Skv;
  const int nkb = (p.Skv + kBN - 1) / kBN;
  const bool sparse = p.blk_idx != nullptr;
  // slots that walk a list of KV tiles (block lists, or the extras' windows)
  const bool listed = sparse || kExtras;

  // ---------------------------------------------------------------- setup
  {
    FA_TR_ROLE(6);
    if (tid == 0) FA_TR(12, 0, 0);
  }
  // The producer thread initialises the barriers and, for dense units, starts
  // the first loads (Q of slot 0, the first K tile, Q of slot 1) before the
  // CTA-wide setup barrier: at a wave's start every CTA loads at once.
  int early = 0;          // producer: ring loads already issued
  bool q_early[2] = {false, false};
  if (warp == 12 && lane == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR_QFULL(t), 1);
      mbar_init(BAR_SFULL(t), 1);
      mbar_init(BAR_OREADY(t), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(BAR_FULL(s), 1);
      mbar_init(BAR_EMPTY(s), 1);
      if (kConvV) mbar_init(BAR_READY(s), 4);   // one arrival per converter warp
    }
    mbar_init(BAR_DRAIN, 1);
    *s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    s_slot[4] = 0;   // first KV tile of the piece
    if (!listed) {
      const int f0 = dense_tiles(qt0, p.n_qt, q_len, kv_len, p.mask);
      const int f1 = dense_tiles(qt1, p.n_qt, q_len, kv_len, p.mask);
      const Piece pc = piece_range(f0, f1, piece, kv_split);
      const int e0 = piece_count(f0, pc), e1 = piece_count(f1, pc);
      s_slot[4] = pc.lo;
      for (int t = 0; t < 2; ++t) {
        if ((t ? e1 : e0) == 0) continue;
        mbar_arrive_expect_tx(BAR_QFULL(t), SM::kQBytes);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sQ + t * SM::kQBytes + bx * (kBM * 128), &p.tm_q, BAR_QFULL(t), 64 * bx,
                      (t ? qt1 : qt0) * kBM, b * p.Hq + (t ? h1 : h0));
        q_early[t] = true;
        if (t == 0) {
          // the first ring load is K tile 0 for Q.K^T(0,0) in every event order
          mbar_arrive_expect_tx(BAR_FULL(0), SM::kStageBytes);
          for (int bx = 0; bx < kBoxes; ++bx)
            tma_load_3d(sStage + bx * (kBN * 128), &p.tm_k, BAR_FULL(0), 64 * bx, pc.lo * kBN,
                        b * p.Hkv + kvh);
          early = 1;
        }
      }
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  // Per-slot KV tile lists and counts.  Dense: the count follows from the
  // lengths and the causal bound.  Block-sparse: warp t compacts the valid
  // slots of its query block (order kept) into s_list[t].
  if (warp < 2) {
    const int t = warp;
    const int qt = t ? qt1 : qt0;
    const int q0 = qt * kBM;
    int n = 0, hilo = 0;
    const bool live = qt < p.n_qt && q0 < q_len && kv_len > 0;
    if (live && !listed) {
      // this slot's tiles of the piece (both slots' counts fix the cuts)
      const int f0 = dense_tiles(qt0, p.n_qt, q_len, kv_len, p.mask);
      const int f1 = dense_tiles(qt1, p.n_qt, q_len, kv_len, p.mask);
      n = piece_count(t ? f1 : f0, piece_range(f0, f1, piece, kv_split));
      const int min_keys = (p.mask == 1) ? min(q0 + 1, kv_len) : kv_len;
      hilo = min_keys < kHiLoKeys;
    } else if (live && kExtras) {
      // the rows' key ranges grow with the row: tiles from the first row's
      // lowest key to the last row's highest
      const int qa = q0, qb = min(q0 + kBM, q_len) - 1;
      const int lo_a = ext_key_lo(p, qa), hi_b = ext_key_hi(p, qb, q_len, kv_len);
      const int t_lo = lo_a / kBN, t_hi = min(nkb, hi_b >= 0 ? hi_b / kBN + 1 : 0);
      n = max(0, t_hi - t_lo);
      for (int e = lane; e < n; e += 32) s_list[t * kMaxSel + e] = t_lo + e;
      // the fewest keys of a row (the count is concave in the row, so at an
      // end).  The cut is twice the plain kernel's: a window gives every row
      // of a tile about the same short length, and with the lazy threshold a
      // 300-key band reached 1.13x the elementwise bound on fp16 P alone.
      // Any row may be short under an explicit mask, and the ALiBi decay
      // leaves few keys that matter (head 0 of 8 at 512 keys: 1.67x); an
      // arbitrary bias tensor may peak any row as well
      const int ka = ext_key_hi(p, qa, q_len, kv_len) - lo_a + 1;
      const int kb = hi_b - ext_key_lo(p, qb) + 1;
      hilo = p.amask != nullptr || p.alibi || p.pse != nullptr || p.keep_thr < 256 ||
             p.dsq != nullptr || min(ka, kb) < 2 * kHiLoKeys;
      if (p.dsv) {
        // the largest d_v over the slot's key tiles
        float dm = 0.f;
        for (int e = lane; e < n; e += 32)
          dm = fmaxf(dm, p.dsv[(long long)(b * p.Hkv + kvh) * p.ds_nbk + t_lo + e]);
        for (int o = 16; o > 0; o >>= 1) dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, o));
        if (lane == 0) s_slot[7 + t] = __float_as_int(dm > 0.f ? dm : 1.f);
      }
    } else if (live && sparse) {
      const int* lst = p.blk_idx + (long long)b * p.blk_stride_b +
                       (long long)(t ? h1 : h0) * p.blk_stride_h + (long long)qt * p.max_sel;
      int keys_lb = 0;
      for (int base = 0; base < p.max_sel; base += 32) {
        const int s = base + lane;
        int e = -1;
        bool ok = false;
        if (s < p.max_sel) {
          e = lst[s];
          ok = e >= 0 && e < nkb && e * kBN < kv_len;
          if (p.mask == 1 && e > qt) ok = false;          // future block: fully masked
        }
        if (ok) {
          const int keys = min(kBN, kv_len - e * kBN);
          const bool diag = (e == qt);
          if (!diag || p.mask == 0) keys_lb += keys;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) s_list[t * kMaxSel + n + __popc(bal & ((1u << lane) - 1))] = e;
        n += __popc(bal);
      }
      for (int o = 16; o > 0; o >>= 1) keys_lb += __shfl_xor_sync(0xffffffffu, keys_lb, o);
      hilo = keys_lb < kHiLoKeys;
    }
    if (lane == 0) {
      s_slot[t] = n;
      s_slot[2 + t] = hilo;
      s_slot[5 + t] = b * p.Hq + (t ? h1 : h0);   // the slot's output plane (for its epilogue)
    }
  }
  named_sync(kBarSetup, kTiledThreads);
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int n0 = s_slot[0], n1 = s_slot[1];
  const int kv_lo = s_slot[4];   // first KV tile of the piece (dense)
  const bool shared_kv = !listed ? (n0 >= 1 && n0 <= n1) : false;
  const WaitCtx wc{s_abort, p.status, p.timeout_ns};

  if (warp < 8) {
    // ============================================================ softmax
    regs_inc<kSoftmaxRegs>();
    FA_TR_ROLE(warp >> 2);
    const int t = warp >> 2;
    const int nt = t ? n1 : n0;
    const int hilo = s_slot[2 + t];
    const int qt = t ? qt1 : qt0;
    const int row = (warp & 3) * 32 + lane;
    const int q0 = qt * kBM;
    const int qi = q0 + row;
    const bool row_valid = qi < q_len;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128u * t + lane_off;
    // scores enter the exponential as s * c - m * c; the extras path scales
    // them to log2 units first (c = 1 there, and m is in log2 units)
    const float c = kExtras ? 1.f : p.scale_log2;
    const uint64_t c2 = f2_pack(c, c);
    // extras: the row's key range, its mask row and the ALiBi slope (log2 units)
    int ek_lo = 0, ek_hi = 0;
    const uint8_t* mrow = nullptr;
    const uint16_t* prow = nullptr;
    float slope2 = 0.f;
    unsigned long long drop_row = 0;   // dropout: grid index of (b, h, row, key 0)
    float ds_q = 1.f;                  // FP8: the query block's dequant scale
    float ds_vmax = 1.f;               // FP8: the largest d_v of the slot's tiles
    if constexpr (kExtras) {
      ek_lo = ext_key_lo(p, qi);
      ek_hi = ext_key_hi(p, qi, q_len, kv_len);
      const int h = t ? h1 : h0;
      if (p.amask)
        mrow = p.amask + b * p.am_sb + h * p.am_sh + (long long)min(qi, p.Sq - 1) * p.am_sq;
      if (p.pse)
        prow = p.pse + b * p.pse_sb + h * p.pse_sh + (long long)min(qi, p.Sq - 1) * p.pse_sq;
      if (p.alibi) slope2 = -exp2f(-8.f * (float)(h + 1) / (float)p.Hq) * 1.4426950408889634f;
      drop_row = ((unsigned long long)(b * p.Hq + h) * p.Sq + min(qi, p.Sq - 1)) * p.Skv;
      if (p.dsq) ds_q = p.dsq[(long long)(b * p.Hq + h) * p.ds_nbq + qt];
      if (p.dsv && nt > 0) ds_vmax = __int_as_float(s_slot[7 + t]);
    }
    float m = -INFINITY, l = 0.f;
    bool dead = false;   // a bounded wait expired: keep the hand-offs, skip the work
    for (int j = 0; j < nt; ++j) {
      // extras: this tile's bytes of the explicit mask, loaded before the S
      // wait (128 keys per row, 16 bytes per load; keys past Skv read none),
      // and its dropout keep bits
      uint4 mbytes[kBN / 16];
      uint32_t dbits[kBN / 32] = {~0u, ~0u, ~0u, ~0u};
      float ds_qk = 1.f, ds_v = 1.f;   // FP8: this key tile's d_q d_k and d_v
      if constexpr (kExtras) {
        if (p.dsq) {
          const long long kb = (long long)(b * p.Hkv + kvh) * p.ds_nbk + s_list[t * kMaxSel + j];
          ds_qk = ds_q * p.dsk[kb];
          if (p.dsv) ds_v = p.dsv[kb] / ds_vmax;
        }
        if (mrow) {
          const int kb0 = s_list[t * kMaxSel + j] * kBN;
#pragma unroll
          for (int q = 0; q < kBN / 16; ++q)
            mbytes[q] = kb0 + 16 * q < p.Skv ? __ldg(reinterpret_cast<const uint4*>(mrow + kb0 + 16 * q))
                                         : make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.keep_thr < 256) {
          // the dropout keep bits of this tile's 128 keys: eight Philox
          // outputs of 16 bytes, one byte per key (bytes of a word low first)
          const int kb0 = s_list[t * kMaxSel + j] * kBN;
          const unsigned long long c0 = p.drop_ctr0 + (drop_row + kb0) / 16;
#pragma unroll
          for (int q = 0; q < kBN / 16; ++q) {
            const unsigned long long cq = c0 + q;
            const uint4 r = philox4x32_10(make_uint4((uint32_t)cq, (uint32_t)(cq >> 32), 0u, 0u),
                                          p.drop_key0, p.drop_key1);
            const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
            uint32_t bits = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              bits |= (((w4[e >> 2] >> (8 * (e & 3))) & 0xFFu) < (uint32_t)p.keep_thr ? 1u : 0u) << e;
            if (q & 1) dbits[q >> 1] |= bits << 16;
            else dbits[q >> 1] = bits;
          }
        }
        if (prow) {
          // the bias row of this tile into L2 (read chunk by chunk below)
          const int kb0 = s_list[t * kMaxSel + j] * kBN;
#pragma unroll
          for (int q = 0; q < kBN / 64; ++q)
            if (kb0 + 64 * q < p.Skv)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(prow + kb0 + 64 * q));
        }
      }
      if (!dead && !__all_sync(0xffffffffu, wait_bar(BAR_SFULL(t), j & 1, wc))) dead = true;
      if (dead) {
        // The MMA issuer waits for one arrival per tile on a hardware barrier.
        // Each arrival, also the one for the tile this warp gave up on, is
        // paced by the issuer's S commit of that tile (a bounded wait past the
        // abort flag): the issuer commits S of tile j only after its "P ready"
        // wait for tile j - 1 completed, so the arrival lands in tile j's
        // generation.  Arriving at once could land it in tile j - 1's, still
        // open, and complete that generation with the wrong set of warps.
        drain_bar(BAR_SFULL(t), j & 1, wc.timeout);
        named_arrive(kBarPReady + t, kPReadyCount);
        continue;
      }
      if (row == 0) FA_TR(1, t, j);
      tc_fence_after();
      // first KV tile of a split launch's piece, re-read from shared memory
      // every tile (a register held across this loop would push the softmax
      // past its budget); unsplit launches skip the load, since shared memory
      // reads wait behind the tensor core's operand traffic
      int kv_first = 0;
      if (kSplit)
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(kv_first) : "r"(smem_u32(s_slot + 4)));
      const int kvt = listed ? s_list[t * kMaxSel + j] : kv_first + j;
      const int kbase = kvt * kBN;
      const bool causal_here = (p.mask == 1) || (p.mask == 2 && kvt == qt);
      const bool need_mask =
          !row_valid || kbase + kBN > kv_len || (causal_here && kbase + kBN - 1 > q0);
      // keys at column >= lim are masked (lim >= kBN when nothing is)
      const int lim = !row_valid ? 0 : min(kv_len - kbase, causal_here ? qi - kbase + 1 : kBN);
      // the whole S row of this thread in registers (4 loads in flight)
      uint32_t su[kBN];
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc)
        tmem_ld32(tS + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&su[32 * cc]));
      tmem_wait_ld();
      float sv[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) sv[i] = __uint_as_float(su[i]);
      if constexpr (kExtras) {
        if (p.dsq) {
          // FP8: the products of the exact x_q values, dequantised
#pragma unroll
          for (int i = 0; i < kBN; ++i) sv[i] *= ds_qk;
        }
        // scores in log2 units, s * scale * log2(e), plus the ALiBi bias
        // -slope_h |i - j| log2(e) (exact integer distances in fp32)
        const float dq = (float)(qi - kbase);
        if (p.alibi == 1) {
#pragma unroll
          for (int i = 0; i < kBN; ++i) sv[i] = fmaf(sv[i], p.scale_log2, slope2 * fabsf(dq - (float)i));
        } else if (p.alibi == 2) {
          // pse_type 3: -slope_h sqrt(|i - j|)
#pragma unroll
          for (int i = 0; i < kBN; ++i) sv[i] = fmaf(sv[i], p.scale_log2, slope2 * sqrtf(fabsf(dq - (float)i)));
        } else if (prow) {
          // the bias tensor, 32 keys (four 16-byte loads) at a time; keys
          // past Skv read none (they are masked below)
          constexpr float kL2e = 1.4426950408889634f;
#pragma unroll
          for (int cc = 0; cc < kBN / 32; ++cc) {
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int col = kbase + 32 * cc + 8 * u;
              w[u] = col < p.Skv ? __ldg(reinterpret_cast<const uint4*>(prow + col)) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t w4[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float b0 = kBF16 ? __uint_as_float(w4[e] << 16) : f16_lo_to_f32(w4[e]);
                const float b1 = kBF16 ? __uint_as_float(w4[e] & 0xFFFF0000u) : f16_hi_to_f32(w4[e]);
                const int i = 32 * cc + 8 * u + 2 * e;
                if (p.pse_type == 1) {
                  sv[i] = (sv[i] + b0) * p.scale_log2;
                  sv[i + 1] = (sv[i + 1] + b1) * p.scale_log2;
                } else {
                  sv[i] = fmaf(sv[i], p.scale_log2, b0 * kL2e);
                  sv[i + 1] = fmaf(sv[i + 1], p.scale_log2, b1 * kL2e);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < kBN; ++i) sv[i] *= p.scale_log2;
        }
        // the mask bytes as bits (a nonzero byte masks its key)
        uint32_t mbits[kBN / 32] = {0u, 0u, 0u, 0u};
        if (mrow) {
#pragma unroll
          for (int q = 0; q < kBN / 16; ++q) {
            const uint32_t w4[4] = {mbytes[q].x, mbytes[q].y, mbytes[q].z, mbytes[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t nz = __vcmpne4(w4[e], 0u) & 0x01010101u;   // 1 per nonzero byte
              mbits[q >> 1] |= ((nz * 0x01020408u) >> 24) << (16 * (q & 1) + 4 * e);
            }
          }
        }
        // keys outside [ek_lo, ek_hi] or masked
        const int lo = ek_lo - kbase, hi = ek_hi - kbase;
        const bool any = lo > 0 || hi < kBN - 1 || (mrow && (mbits[0] | mbits[1] | mbits[2] | mbits[3]));
        if (__any_sync(0xffffffffu, any)) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (i < lo || i > hi || ((mbits[i >> 5] >> (i & 31)) & 1u)) sv[i] = -INFINITY;
        }
      } else if (__any_sync(0xffffffffu, need_mask)) {
        // Warp-uniform decisions per 32-column chunk: chunks below every row's
        // limit stay, chunks above every limit are cleared, and only a chunk
        // that straddles the warp's limits (the diagonal block of a causal
        // tile, a ragged tail) is masked element by element.
        const int lim_lo = __reduce_min_sync(0xffffffffu, lim);
        const int lim_hi = __reduce_max_sync(0xffffffffu, lim);
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          const bool clear = 32 * cc >= lim_hi;
          const bool part = !clear && 32 * cc + 32 > lim_lo;
          if (clear) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[32 * cc + i] = -INFINITY;
          }
          if (part) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * cc + i >= lim) sv[32 * cc + i] = -INFINITY;
          }
        }
      }
      const float mb = row_max(sv);
      const float m_new = fmaxf(m, mb);
      float m_use = m_new, alpha = 1.f;
      if (m != -INFINITY) {
        const float step = (m - m_new) * c;     // <= 0, log2 units of scaled scores
        if (step >= -p.threshold) {
          m_use = m;                            // keep the (possibly stale) max
        } else {
          alpha = ex2_approx(step);
        }
      }
      const float neg = (m_use == -INFINITY) ? 0.f : -m_use * c;
      const uint64_t neg2 = f2_pack(neg, neg);
      // p = exp2(s c - m c); P (fp16) written over S (all of S is already in
      // registers), with the hi+lo split (second fp16 term p - fp16(p) in
      // columns 64..127) for rows that see few keys
      uint64_t sum2[2] = {0ull, 0ull};
      // (two copies of the loop: a hi+lo test inside it costs more instructions
      // than the exponentials themselves)
      if (!hilo) {
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t ph[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(sv[32 * cc + 2 * i], sv[32 * cc + 2 * i + 1]), c2, neg2), a0, a1);
            a0 = ex2_approx(a0);
            a1 = ex2_approx(a1);
            sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(a0, a1));
            ph[i] = pack_f16x2(a0, a1);
          }
          tmem_st16(tS + 16 * cc, ph);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(sv[32 * cc + 2 * i], sv[32 * cc + 2 * i + 1]), c2, neg2), a0, a1);
            a0 = ex2_approx(a0);
            a1 = ex2_approx(a1);
            sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(a0, a1));
            if constexpr (kExtras) {
              // dropout: the row sum keeps every p, the P.V operand only the kept
              // ones (the 1 / keep_prob factor is applied with 1 / l)
              // (FP8: d_v of the key tile joins the P.V operand)
              a0 = ((dbits[cc] >> (2 * i)) & 1u) ? a0 * ds_v : 0.f;
              a1 = ((dbits[cc] >> (2 * i + 1)) & 1u) ? a1 * ds_v : 0.f;
            }
            ph[i] = pack_f16x2(a0, a1);
            pl[i] = pack_f16x2(a0 - f16_lo_to_f32(ph[i]), a1 - f16_hi_to_f32(ph[i]));
          }
          tmem_st16(tS + 16 * cc, ph);
          tmem_st16(tS + 64 + 16 * cc, pl);
        }
      }
      float r0, r1, r2, r3;
      f2_unpack(sum2[0], r0, r1);
      f2_unpack(sum2[1], r2, r3);
      l = __fmaf_rn(alpha, l, (r0 + r1) + (r2 + r3));   // (one rounding in every build)
      m = m_use;
      // O_t *= alpha for the rows whose max moved.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // (the previous P.V product into O_t has completed: the commit that
        // signalled S for this tile tracks every earlier MMA of the issuer)
        // (all of the row in flight at once: the S row's registers are free here)
        const uint32_t tO = tmem + 256u + 128u * t + lane_off;
        const uint64_t a2 = f2_pack(alpha, alpha);
        uint32_t r[Dv];
#pragma unroll
        for (int cc = 0; cc < Dv / 32; ++cc)
          tmem_ld32(tO + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * cc]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < Dv / 2; ++i) {
          float x0, x1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), a2), x0, x1);
          r[2 * i] = __float_as_uint(x0);
          r[2 * i + 1] = __float_as_uint(x1);
        }
#pragma unroll
        for (int cc = 0; cc < Dv / 32; ++cc)
          tmem_st32(tO + 32 * cc, *reinterpret_cast<const uint32_t(*)[32]>(&r[32 * cc]));
      }
      tmem_wait_st();
      tc_fence_before();
      if (row == 0) FA_TR(2, t, j);
      // P_t (and the rescaled O_t) ready: hardware barrier to the MMA issuer
      named_arrive(kBarPReady + t, kPReadyCount);
    }
    // ---- epilogue of slot t, by its own threads (m and l are in registers):
    // O / l and the LSE.  O_t is complete once the slot's last P.V has
    // finished; the slot's Q buffer (its last reader, Q.K^T, finished before
    // that P.V) stages the output tile, which the slot's threads then copy to
    // memory row by row (each warp store covers 512 contiguous bytes).  Plain
    // stores let the CTA retire without waiting for them to drain.
    if (qt < p.n_qt) {
      bool skip = false;
      if (nt > 0) {
        const bool ok = !dead && __all_sync(0xffffffffu, wait_bar(BAR_OREADY(t), 0, wc));
        // one decision for the slot's four warps, so that none waits at the
        // staging barrier below for a warp that gave up
        skip = named_or(kBarEpi + t, kBM, !ok);
        if (!skip) tc_fence_after();
      }
      if (!skip) {
        // the slot's (batch, head) plane, re-read here rather than held in a
        // register across the tile loop
        int plane;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(plane)
                     : "r"(((smem_u32(smem_raw) + 1023u) & ~1023u) + SM::kMiscOff + 8 + 4 * (5 + t)));
        const bool write = qi < p.Sq;
        // (extras: the dropout factor and the FP8 V scale join 1 / l; the
        // scale is re-read here rather than held across the loop)
        float vmax = 1.f;
        if constexpr (kExtras) {
          if (p.dsv && nt > 0)
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=f"(vmax)
                         : "r"(((smem_u32(smem_raw) + 1023u) & ~1023u) + SM::kMiscOff + 8 + 4 * (7 + t)));
        }
        const float inv_l = (l > 0.f) ? (kExtras ? vmax / (l * p.keep_prob) : 1.f / l) : 0.f;
        const uint32_t tO = tmem + 256u + 128u * t + lane_off;
        const uint32_t stage = ((smem_u32(smem_raw) + 1023u) & ~1023u) + SM::kQOff + t * SM::kQBytes;
        const size_t rows_all = (size_t)p.B * p.Hq * p.Sq;
        const size_t rr = (size_t)plane * p.Sq + (write ? qi : 0);
        // this CTA's piece of a split unit (recomputed: nothing held across the loop)
        const int my_piece = kSplit ? (int)(blockIdx.x % (unsigned)p.kv_split) : 0;
        // O in halves of 64 columns: TMEM -> registers, O / l, out
#pragma unroll 1
        for (int hh = 0; hh < Dv / 64; ++hh) {
          uint32_t r[64];
          if (nt > 0) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)   // warp-collective: all lanes, even rows past Sq
              tmem_ld32(tO + 64 * hh + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * cc]));
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) r[i] = 0;
          }
          const uint64_t il2 = f2_pack(inv_l, inv_l);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), il2), x0, x1);
            r[2 * i] = __float_as_uint(x0);
            r[2 * i + 1] = __float_as_uint(x1);
          }
          if (kSplit) {
            // one piece of a split unit: its O / l in fp32 for the merge kernel
            float4* dst = reinterpret_cast<float4*>(p.part_o + ((size_t)my_piece * rows_all + rr) * Dv + 64 * hh);
            if (write) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                     __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            }
          } else {
            // O / l rounded to o's type, staged in the slot's Q buffer: row-major,
            // 16-byte chunk c of row i at i * 2 Dv + ((c ^ i) & 15) * 16 (the XOR
            // spreads the 32 rows of one warp store over the banks)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {   // 16-byte chunks of eight outputs
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a0 = __uint_as_float(r[8 * c8 + 2 * e]);
                const float a1 = __uint_as_float(r[8 * c8 + 2 * e + 1]);
                w[e] = kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
              }
              const int c = 8 * hh + c8;
              st_shared_v4(stage + row * (2 * Dv) + (((c ^ row) & (Dv / 8 - 1)) << 4),
                           make_uint4(w[0], w[1], w[2], w[3]));
            }
            if (p.o_lo && write) {
              // o's rounding residual (only when asked for), straight to memory
              uint4* dst_lo = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o_lo) + (rr * Dv + 64 * hh) * 2);
#pragma unroll
              for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float a0 = __uint_as_float(r[8 * c8 + 2 * e]);
                  const float a1 = __uint_as_float(r[8 * c8 + 2 * e + 1]);
                  wl[e] = pack_residual_x2(a0, a1, kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1), kBF16);
                }
                dst_lo[c8] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
              }
            }
          }
        }
        if (kSplit) {
          if (write)
            p.part_lse[(size_t)my_piece * rows_all + rr] = (l > 0.f) ? __fmaf_rn(m, p.scale, __logf(l)) : -INFINITY;
        } else {
          if (write)
            p.lse[rr] = (l > 0.f) ? __fmaf_rn(m, kExtras ? 0.6931471805599453f : p.scale, __logf(l))
                                  : INFINITY;
          named_sync(kBarEpi + t, kBM);   // the slot's four warps staged their rows
          // copy-out: the slot's 128 threads walk the tile in 16-byte chunks,
          // consecutive threads on consecutive chunks of a row
          constexpr int kChunks = Dv / 8;                // per row
          constexpr int kRowsPerPass = kBM * 16 / (2 * Dv);
          const int c = row % kChunks;
          const int i0 = row / kChunks;
          const int rows_left = p.Sq - q0;               // rows past Sq are not written
          uint8_t* out = static_cast<uint8_t*>(p.o) + ((size_t)plane * p.Sq + q0) * (2 * Dv) + c * 16;
#pragma unroll
          for (int k = 0; k < kBM / kRowsPerPass; k += 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = i0 + (k + u) * kRowsPerPass;
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                           : "r"(stage + i * (2 * Dv) + (((c ^ i) & (kChunks - 1)) << 4)));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = i0 + (k + u) * kRowsPerPass;
              if (i < rows_left) *reinterpret_cast<uint4*>(out + (size_t)i * (2 * Dv)) = v[u];
            }
          }
        }
        if (row == 0) FA_TR(11, t, 0);
      }
    }
  } else if (warp < 12) {
    // ============================================================ V converter
    regs_dec<kCorrRegs>();
    FA_TR_ROLE(2);
    if constexpr (kConvV) {
      // Every ring load in the producer's order: wait until it landed; a V tile
      // is converted bf16 -> fp16 in place (exact for 2^-14 <= |v| <= 65504;
      // larger magnitudes become inf and set the range bit), then the load is
      // released to the MMA side.
      int ld = 0;
      bool dead = false;
      uint32_t vmax = 0;
      const int ne = num_events(n0, n1);
      for (int e = 0; e < ne; ++e) {
        const Event ev = event_at(e, n0, n1, shared_kv);
        if (!ev.valid || !ev.load) continue;
        const int s = ld % NS;
        const uint32_t f = ld / NS;
        ++ld;
        if (!dead && !__all_sync(0xffffffffu, wait_bar(BAR_FULL(s), f & 1, wc))) dead = true;
        if (!dead && ev.pv) {
          uint4* tile = reinterpret_cast<uint4*>(smem + SM::kStageOff + s * SM::kStageBytes);
#pragma unroll 4
          for (int i = tid - 256; i < SM::kStageBytes / 16; i += 128) {
            uint4 w = tile[i];
            uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              vmax = max_u16x2(vmax, ww[q] & 0x7FFF7FFFu);
              ww[q] = pack_f16x2(__uint_as_float(ww[q] << 16), __uint_as_float(ww[q] & 0xFFFF0000u));
            }
            tile[i] = w;
          }
          fence_proxy_async_smem();   // generic-proxy writes -> tensor core reads
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_READY(s));
      }
      if ((vmax & 0xFFFFu) > 0x477Fu || (vmax >> 16) > 0x477Fu) atomicOr(p.status, kStatusRange);
    }
  } else if (warp == 12) {
    // ============================================================ producer
    regs_dec<kOtherRegs>();
    FA_TR_ROLE(3);
    if (lane == 0) {
      for (int t = 0; t < 2; ++t) {
        if ((t ? n1 : n0) == 0 || q_early[t]) continue;
        mbar_arrive_expect_tx(BAR_QFULL(t), SM::kQBytes);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sQ + t * SM::kQBytes + bx * (kBM * 128), &p.tm_q, BAR_QFULL(t), 64 * bx,
                      (t ? qt1 : qt0) * kBM, b * p.Hq + (t ? h1 : h0));
      }
      int ld = 0;
      const int ne = num_events(n0, n1);
      for (int e = 0; e < ne; ++e) {
        const Event ev = event_at(e, n0, n1, shared_kv);
        if (!ev.valid || !ev.load) continue;
        const int s = ld % NS;
        const uint32_t f = ld / NS;
        ++ld;
        if (ld <= early) continue;   // issued before the setup barrier
        // the stage's readers are done, and its previous copy has landed (its
        // readers waited for it on the normal path, but after a give-up they
        // release the stage without waiting): at most one copy is ever in
        // flight per stage, so each phase of its barrier belongs to one copy
        if (!wait_bar(BAR_EMPTY(s), (f & 1) ^ 1, wc) ||
            (f > 0 && !wait_bar(BAR_FULL(s), (f - 1) & 1, wc))) {
          --ld;   // not issued: ld counts the loads in flight or landed
          break;
        }
        const int kvt = listed ? s_list[ev.t * kMaxSel + ev.j] : kv_lo + ev.j;
        FA_TR(5, ev.t, ev.j);
        mbar_arrive_expect_tx(BAR_FULL(s), SM::kStageBytes);
        const CUtensorMap* tm = ev.pv ? &p.tm_v : &p.tm_k;
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sStage + s * SM::kStageBytes + bx * (kBN * 128), tm, BAR_FULL(s), 64 * bx,
                      kvt * kBN, b * p.Hkv + kvh);
      }
      // Every copy lands before the CTA's shared memory goes away: the last
      // load of each stage and the Q tiles, whether or not some role gave up
      // (a role may give up after this point, with a copy still in flight).
      // On the normal path these phases completed long ago (each is its
      // stage's last), so the waits pass at once.
      for (int i = (ld > NS ? ld - NS : 0); i < ld; ++i)
        drain_bar(BAR_FULL(i % NS), (i / NS) & 1, wc.timeout);
      for (int t = 0; t < 2; ++t)
        if ((t ? n1 : n0) > 0) drain_bar(BAR_QFULL(t), 0, wc.timeout);
    }
    __syncwarp();
  } else if (warp == 13 || warp == 14) {
    // ============================================================ MMA issue
    // Work is handed out as "groups": QK(0,0), QK(1,0), then per iteration j
    // the pairs [PV(0,j) QK(0,j+1)] and [PV(1,j) QK(1,j+1)].  Warp 14 (the
    // scheduler) waits on the TMA mbarriers a group depends on and releases the
    // group to warp 13 (the issuer) through hardware named barriers, running up
    // to two groups ahead: for every group with a P.V it arrives on the slot's
    // "P ready" barrier, where the softmax warps arrive too, so the issuer
    // waits once per group.  The issuer never polls shared memory, which the
    // tensor core's operand reads keep busy.
    regs_dec<kOtherRegs>();
    FA_TR_ROLE(warp == 13 ? 4 : 5);
    const bool issuer = (warp == 13);
    const int hilo0 = s_slot[2], hilo1 = s_slot[3];
    const uint64_t q_desc0 = sw128_desc(sQ, 16, 1024);               // K-major Q
    const uint64_t k_desc0 = sw128_desc(sStage, 16, 1024);           // K-major K
    const uint64_t v_desc0 = sw128_desc(sStage, kBN * 128, 1024);    // MN-major V
    const int nmax = n0 > n1 ? n0 : n1;
    const int ngroups = nmax > 0 ? 2 + 2 * nmax : 0;
    if (!issuer) {
      // ---- scheduler: walks the groups in order, waits for the TMA copies a
      // group reads and releases it: groups 0 and 1 (Q.K^T only) on named
      // barrier 1 + g, every later group on the slot's "P ready" barrier,
      // which the softmax warps of the slot complete as well
      int ld = 0;            // ring loads consumed so far (independent K/V sequences)
      bool aborted = false;
#pragma unroll 1
      for (int g = 0; g < ngroups; ++g) {
        const int t = g < 2 ? g : ((g - 2) & 1);
        const int jpv = g < 2 ? -1 : ((g - 2) >> 1);         // P.V tile (none in groups 0, 1)
        const int jqk = g < 2 ? 0 : jpv + 1;                 // Q.K^T tile
        const int nt = t ? n1 : n0;
        const bool pv_valid = jpv >= 0 && jpv < nt;
        const bool qk_valid = jqk < nt;
        // with shared K/V, slot 1 reuses slot 0's tiles and the load order is
        // K_0 V_0 K_1 V_1 ...; otherwise every event loads its own tile, in order
        const bool pv_load = pv_valid && (!shared_kv || t == 0 || jpv >= n0);
        const bool qk_load = qk_valid && (!shared_kv || t == 0 || jqk >= n0);
        int lpv, lqk;
        if (shared_kv) {
          lpv = 2 * jpv + 1;
          lqk = 2 * jqk;
        } else {
          lpv = ld;
          lqk = ld + (pv_load ? 1 : 0);
          ld += (pv_load ? 1 : 0) + (qk_load ? 1 : 0);
        }
        const uint32_t sv_ = (uint32_t)lpv % NS, sk_ = (uint32_t)lqk % NS;
        // issuer finished group g-2 (a group with work: groups 0 and 1, or a
        // P.V at tile jpv - 1 < nt; an empty group arrives nowhere)
        if (g >= 2 && (g < 4 || jpv <= nt)) named_sync(3 + (g & 1), 64);
        if (lane == 0 && !aborted) {
          if (pv_load && !wait_bar(BAR_READY(sv_), (lpv / NS) & 1, wc)) aborted = true;
          if (!aborted && qk_load && !wait_bar(BAR_READY(sk_), (lqk / NS) & 1, wc)) aborted = true;
          if (!aborted && qk_valid && jqk == 0 && !wait_bar(BAR_QFULL(t), 0, wc)) aborted = true;
        }
        aborted = __shfl_sync(0xffffffffu, aborted, 0);
        // (after a timeout every group is still released; the issuer then runs
        // on stale operands, which is harmless: the status word already
        // reports the failure and nothing waits on the results)
        if (g < 2) {
          named_arrive(1 + g, 64);
        } else if (pv_valid) {
          named_arrive(kBarPReady + t, kPReadyCount);
        }
      }
      // the issuer's last two "group issued" arrivals: groups (0, nmax - 1)
      // and (1, nmax - 1), each only if its slot has a P.V there
      if (nmax > 0 && n0 == nmax) named_sync(3, 64);
      if (nmax > 0 && n1 == nmax) named_sync(4, 64);
    } else {
      // ---- issuer: the same groups, two per step (slot 0, slot 1) so that
      // everything that depends on the slot is fixed at compile time.  The
      // whole warp runs the issue code (warp-uniform branches only); the
      // elected lane's predicate lets exactly one copy of each tcgen05
      // instruction through (always the same lane: a commit tracks the MMAs
      // of the thread that issues it).
      const uint32_t lead = elect_lane();
      int ld = 0;
      auto group = [&](auto slot, int jpv) {
        constexpr int t = decltype(slot)::value;
        const int nt = t ? n1 : n0;
        const int jqk = jpv + 1;
        const bool pv_valid = jpv >= 0 && jpv < nt;
        const bool qk_valid = jqk < nt;
        // A group past the slot's last tile has no work (no P.V, hence no
        // Q.K^T) and hands nothing off: its "group issued" arrival could
        // otherwise follow the previous one on the same barrier before the
        // scheduler has consumed that one, completing the barrier's generation
        // with the wrong pair and leaving the scheduler waiting forever.
        if (jpv >= 0 && !pv_valid) return;
        int lpv, lqk;
        if (shared_kv) {
          lpv = 2 * jpv + 1;
          lqk = 2 * jqk;
        } else {   // every valid event loads its own tile
          lpv = ld;
          lqk = ld + (pv_valid ? 1 : 0);
          ld += (pv_valid ? 1 : 0) + (qk_valid ? 1 : 0);
        }
        const uint32_t sv_ = (uint32_t)lpv % NS, sk_ = (uint32_t)lqk % NS;
        if (jpv < 0) {
          named_sync(1 + t, 64);   // the first K tile and Q_t landed
        } else if (pv_valid) {
          // P_t of tile jpv written by the four softmax warps of slot t (a
          // softmax warp that gave up still arrives once per tile, paced by
          // the S commits, so this wait always ends) and the group's copies
          // landed (the scheduler's arrival)
          named_sync(kBarPReady + t, kPReadyCount);
          tc_fence_after();
        }
        constexpr uint32_t kS = 128u * t, kO = 256u + 128u * t;
        // the group's operand bases pass an empty asm, so that the compiler
        // derives each MMA's operands here instead of keeping those of every
        // MMA of both slots live across the loop
        uint32_t tb = tmem;
        uint64_t vb = v_desc0, kb = k_desc0, qb = q_desc0;
        asm volatile("" : "+r"(tb), "+l"(vb), "+l"(kb), "+l"(qb));
        if (pv_valid) {
          if (lead) FA_TR(7, t, jpv);
          const uint64_t vd = vb + ((sv_ * SM::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_if(tb + kO, tb + kS + 8 * kk, vd + (kk * 2048 >> 4), kIdescPV,
                      (jpv > 0 || kk > 0) ? 1u : 0u, lead);
          if (t ? hilo1 : hilo0) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_if(tb + kO, tb + kS + 64 + 8 * kk, vd + (kk * 2048 >> 4), kIdescPV, 1u,
                        lead);
          }
          // O_t is read only by the epilogue, after the slot's last P.V
          if (jpv == nt - 1) mma_commit_if(BAR_OREADY(t), lead);
          // V's last reader is slot 1 (shared K/V) or this slot
          if (!shared_kv || t == 1) mma_commit_if(BAR_EMPTY(sv_), lead);
        }
        if (qk_valid) {
          // S_t is free: the softmax read it before signalling P ready, which
          // was waited on (and fenced) before the previous P.V
          if (lead) FA_TR(6, t, jqk);
          const uint64_t qd = qb + ((t * SM::kQBytes) >> 4);
          const uint64_t kd = kb + ((sk_ * SM::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKSteps; ++kk) {
            const uint32_t off16 = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
            mma_ss_if(tb + kS, qd + off16, kd + off16, kIdescQK, kk > 0, lead);
          }
          mma_commit_if(BAR_SFULL(t), lead);
          if (!shared_kv || t == 1) mma_commit_if(BAR_EMPTY(sk_), lead);
        }
        __syncwarp();
        named_arrive(3 + t, 64);   // group issued (its index has the slot's parity)
      };
      if (ngroups > 0) {
        group(std::integral_constant<int, 0>{}, -1);
        group(std::integral_constant<int, 1>{}, -1);
#pragma unroll 1
        for (int j = 0; j < nmax; ++j) {
          group(std::integral_constant<int, 0>{}, j);
          group(std::integral_constant<int, 1>{}, j);
        }
      }
    }
    // every MMA has finished before TMEM is released
    if (issuer && elect_lane() && n0 + n1 > 0) {
      mma_commit(BAR_DRAIN);
      drain_bar(BAR_DRAIN, 0, wc.timeout);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  {
    FA_TR_ROLE(7);
    if (tid == 0) FA_TR(13, 0, 0);
  }
}

}  // namespace fa
