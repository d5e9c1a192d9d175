// Attention backward for sm_103a: dQ, dK, dV of the dense forward (causal or
// not, per-batch lengths, GQA), D = Dv = 128, fp16 tensor-core operands.
//
// The steps are those of the BSA PyPTO implementation notes' backward
// (section 3.2 "Core design strategies": S and P are not stored, P is
// recomputed as exp(scale * S - LSE) from the forward's LSE; section 8.4:
// d_row = rowsum(dO * O) is computed once beforehand; section 1: dV carries
// no scale, dQ and dK are multiplied by it):
//   dV = P^T dO,   dS = P * (dO V^T - d_row),   dQ = scale dS K,   dK = scale dS^T Q
// Two kernels, as the notes' two phases (dK / dV, then dQ), without atomics:
//   fa_bwd_dkdv_kernel  one CTA per (batch, KV head, 128-key tile); K and V stay
//                       in shared memory while the query tiles that see the keys
//                       (of every head of the GQA group) stream through
//   fa_bwd_dq_kernel    one CTA per (batch, head, 128-row query tile); Q and dO
//                       stay while the key tiles stream through
// Warps: 0-3 elementwise (one thread per row of the transposed or plain score
// tile), then the epilogue; 4 TMA producer; 5 TMEM allocator and MMA issuer.
// Every hand-off is an mbarrier with a bounded wait.
//
// Precision: every MMA runs on fp16 operands (bf16 inputs arrive as fp16
// copies); P and dS are fp16, and on query rows with fewer than kBwdHiLoKeys
// valid keys a second fp16 term x - fp16(x) doubles the product (the
// forward's hi + lo split).  d_row should come from O + o_lo, the forward's
// output and its rounding residual: from the rounded output alone the dpsum
// error dominates dQ and dK on causal problems.
#pragma once
#include "fa_tiled.cuh"

namespace fa {

constexpr int kBwdThreads = 192;
// query rows with fewer keys than this take the hi + lo split of P and dS
// (twice the forward's threshold: the backward's fp16 dS rounding reaches
// the rows just above the threshold, and 512 keeps about half the bound free)
constexpr int kBwdHiLoKeys = 512;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // fp16; boxes of 64 columns x 128 rows, 128-byte swizzle
  const float* lse;     // [B*Hq*Sq]: the forward's LSE (+inf on rows without keys)
  const float* d_row;   // [B*Hq*Sq]: rowsum(dO * O)
  void* dq;             // [B, Hq, Sq, 128]  (output type: bf16 or fp16)
  void* dk;             // [B, Hkv, Skv, 128]
  void* dv;             // [B, Hkv, Skv, 128]
  const int* seqlens;
  int B, Hq, Hkv, Sq, Skv, G, n_qt, n_kt;
  int causal;
  float scale, scale_log2;
  long long timeout_ns;
  int* status;
};

// Shared memory (offsets from a 1024-byte aligned base): two resident tiles,
// two stages of two tiles, the staged per-query values of two steps, barriers.
struct BwdSmem {
  static constexpr int kTile = 128 * 128 * 2;            // a 128 x 128 fp16 tile (two boxes)
  static constexpr int kRes0 = 0;
  static constexpr int kRes1 = kTile;
  static constexpr int kStage = 2 * kTile;                // stage s at kStage + 2 s kTile
  static constexpr int kRowOff = kStage + 4 * kTile;      // [2 steps][LSE*log2(e), d_row][128]
  static constexpr int kBarOff = kRowOff + 2 * 2 * 128 * 4;
  // barriers: resident, full[2], empty[2], s_ready, p_ready, acc, drain
  static constexpr int kNumBars = 9;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

constexpr uint32_t kIdescBwdSS = idesc_f16(128, 128, false, false);   // fp16 A, B K-major
constexpr uint32_t kIdescBwdTS = idesc_f16(128, 128, false, true);    // fp16, B MN-major

// A 128 x 128 fp16 tile as two 64-column boxes (rows past the tensor read as 0).
__device__ __forceinline__ void bwd_load_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar,
                                              int row0, int plane) {
  tma_load_3d(dst, tm, bar, 0, row0, plane);
  tma_load_3d(dst + 128 * 128, tm, bar, 64, row0, plane);
}
// Byte offset (>> 4) of k-step kk (16 elements) in a K-major tile.
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
  return (uint32_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
}
// ... and in an MN-major tile (16 rows of 128 bytes per k-step).
__device__ __forceinline__ uint32_t mnmajor_step(int kk) { return (uint32_t)((kk * 2048) >> 4); }

// Lane-0 bounded wait, result broadcast to the warp (the warp stays converged).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, WaitCtx wc) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, wc);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Rows of a query tile with fewer than kBwdHiLoKeys valid keys take the hi + lo split.
__device__ __forceinline__ bool bwd_hilo(int q0, int kv_len, int causal) {
  return (causal ? min(q0 + 1, kv_len) : kv_len) < kBwdHiLoKeys;
}

// P (fp32, 128 values of one row) into TMEM as fp16 at `t`, and the
// residual terms at t + 64 when `hilo`.
__device__ __forceinline__ void bwd_store_p(uint32_t t, const float (&pr)[128], bool hilo) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t ph[16], pl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float a0 = pr[32 * cc + 2 * i], a1 = pr[32 * cc + 2 * i + 1];
      ph[i] = pack_f16x2(a0, a1);
      pl[i] = pack_f16x2(a0 - f16_lo_to_f32(ph[i]), a1 - f16_hi_to_f32(ph[i]));
    }
    tmem_st16(t + 16 * cc, ph);
    if (hilo) tmem_st16(t + 64 + 16 * cc, pl);
  }
}

// dS = P * (dP - d) for one row: dP read from TMEM at `t` in 32-column chunks,
// dS written back over it as fp16 (the high terms right away, over columns
// already read; the residual terms at t + 64 once the whole row is read).
// `drow(i)` gives d for column i.
template <typename DRow>
__device__ __forceinline__ void bwd_store_ds(uint32_t t, const float (&pr)[128], bool hilo,
                                             DRow drow) {
  uint32_t dl[64];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t du[32];
    tmem_ld32(t + 32 * cc, du);
    tmem_wait_ld();
    uint32_t dh[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c0 = 32 * cc + 2 * i;
      const float x0 = pr[c0] * (__uint_as_float(du[2 * i]) - drow(c0));
      const float x1 = pr[c0 + 1] * (__uint_as_float(du[2 * i + 1]) - drow(c0 + 1));
      dh[i] = pack_f16x2(x0, x1);
      dl[16 * cc + i] = pack_f16x2(x0 - f16_lo_to_f32(dh[i]), x1 - f16_hi_to_f32(dh[i]));
    }
    tmem_st16(t + 16 * cc, dh);   // over dP columns [16 cc, 16 cc + 16): read in this or an earlier chunk
  }
  if (hilo) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      tmem_st16(t + 64 + 16 * cc, *reinterpret_cast<const uint32_t(*)[16]>(&dl[16 * cc]));
  }
}

// One row of a 128-column fp32 accumulator (TMEM at `t`) times `mul`, stored
// as 128 bf16 / fp16 values at `dst` (zeros when !have); skipped when !write.
template <bool kBF16>
__device__ __forceinline__ void bwd_store_row(uint32_t t, bool have, float mul, bool write,
                                              uint8_t* dst) {
#pragma unroll 1
  for (int cc = 0; cc < 8; ++cc) {
    uint32_t r[16];
    if (have) {
      tmem_ld16(t + 16 * cc, r);   // warp-collective
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = 0;
    }
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float a0 = __uint_as_float(r[2 * e]) * mul, a1 = __uint_as_float(r[2 * e + 1]) * mul;
      w[e] = kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
    }
    if (write) {
      reinterpret_cast<uint4*>(dst)[2 * cc] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst)[2 * cc + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// The CTA's shared-memory base, barriers and flags (the same plan in both
// kernels): resident, full[2], empty[2], s_ready, p_ready, acc, drain.
struct BwdCta {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t bar0;
  uint32_t* s_tmem;
  volatile int* s_abort;
  __device__ uint32_t res() const { return bar0; }
  __device__ uint32_t full(int s) const { return bar0 + 8u + 8u * s; }
  __device__ uint32_t empty(int s) const { return bar0 + 24u + 8u * s; }
  __device__ uint32_t s_ready() const { return bar0 + 40u; }
  __device__ uint32_t p_ready() const { return bar0 + 48u; }
  __device__ uint32_t acc() const { return bar0 + 56u; }
  __device__ uint32_t drain() const { return bar0 + 64u; }
};

// Setup common to both kernels: barriers (warp 4, lane 0), the 512 TMEM
// columns (warp 5), then a CTA barrier.  Returns the TMEM base.
__device__ __forceinline__ uint32_t bwd_setup(BwdCta& c, uint8_t* smem_raw) {
  c.smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  c.sbase = smem_u32(c.smem);
  c.bar0 = c.sbase + BwdSmem::kBarOff;
  c.s_tmem = reinterpret_cast<uint32_t*>(c.smem + BwdSmem::kMiscOff);
  c.s_abort = reinterpret_cast<volatile int*>(c.smem + BwdSmem::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 4 && lane == 0) {
    mbar_init(c.res(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(c.full(s), 1);
      mbar_init(c.empty(s), 1);
    }
    mbar_init(c.s_ready(), 1);
    mbar_init(c.p_ready(), 4);   // lane 0 of each elementwise warp
    mbar_init(c.acc(), 1);
    mbar_init(c.drain(), 1);
    *c.s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(c.s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  return *c.s_tmem;
}

// Teardown: every role done (the MMA warp drained its products), TMEM freed.
__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dK and dV of one 128-key tile.  TMEM: S^T / P^T at column 0, dP^T / dS^T at
// 128, dV at 256, dK at 384 (rows = keys).
// With GQA (G > 1) every step takes the hi + lo split: dK and dV then sum the
// fp16 roundings of P and dS over the group's heads, and long rows' terms
// alone pass the elementwise bound where the result nearly cancels.
template <bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using SM = BwdSmem;
  extern __shared__ uint8_t smem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heaviest key tiles (the first ones, under a causal mask) first
  const int per_kt = p.B * p.Hkv;
  const int kt = blockIdx.x / per_kt;
  const int bk = blockIdx.x - kt * per_kt;
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int q_len = p.seqlens ? min(p.seqlens[b], p.Sq) : p.Sq;
  const int kv_len = p.seqlens ? min(p.seqlens[b], p.Skv) : p.Skv;
  const int k0 = kt * 128;
  // the query tiles that see the tile's keys: [qt_lo, qt_hi), for every head of the group
  const int qt_hi = (q_len + 127) / 128;
  const int qt_lo = p.causal ? kt : 0;
  const int nq = (k0 < kv_len && qt_hi > qt_lo) ? qt_hi - qt_lo : 0;
  const int nsteps = nq * p.G;   // step n: head kvh * G + n / nq, query tile qt_lo + n % nq

  BwdCta cta;
  const uint32_t tmem = bwd_setup(cta, smem_raw);
  const uint32_t sbase = cta.sbase;
  const uint32_t BAR_RES = cta.res(), BAR_S = cta.s_ready(), BAR_P = cta.p_ready(),
                 BAR_ACC = cta.acc(), BAR_DRAIN = cta.drain();
  auto BAR_FULL = [=](int s) { return cta.full(s); };
  auto BAR_EMPTY = [=](int s) { return cta.empty(s); };
  volatile int* s_abort = cta.s_abort;
  const WaitCtx wc{s_abort, p.status, p.timeout_ns};

  if (warp < 4) {
    // ============================================================ elementwise
    const int row = warp * 32 + lane;   // key row of the tile
    const int kj = k0 + row;
    const bool key_ok = kj < kv_len;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off, tD = tmem + 128u + lane_off;
    bool dead = false;
#pragma unroll 1
    for (int n = 0; n < nsteps; ++n) {
      const int g = n / nq, qt = qt_lo + n - g * nq;
      const int h = kvh * p.G + g;
      const int q0 = qt * 128;
      // this step's per-query values: LSE in log2 units (+inf past the rows)
      // and d_row (0 past the rows), one per thread, read by all
      float* buf = reinterpret_cast<float*>(cta.smem + SM::kRowOff) + (n & 1) * 256;
      {
        const int qi = q0 + row;
        const bool live = qi < q_len;
        const size_t r = (size_t)(b * p.Hq + h) * p.Sq + (live ? qi : 0);
        const float l = live ? p.lse[r] : INFINITY;
        buf[row] = (l == INFINITY) ? INFINITY : l * kLog2e;
        buf[128 + row] = live ? p.d_row[r] : 0.f;
      }
      named_sync(1, 128);   // the four elementwise warps (same step count)
      if (!dead && !__all_sync(0xffffffffu, wait_bar(BAR_S, n & 1, wc))) dead = true;
      if (!dead) {
        tc_fence_after();
        const bool hilo = p.G > 1 || bwd_hilo(q0, kv_len, p.causal);   // GQA: every row (see above)
        const int lim = p.causal ? kj - q0 : -1;   // query column i sees the key iff i >= lim
        float pr[128];
        {
          uint32_t su[128];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            tmem_ld32(tS + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&su[32 * cc]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            const float e = ex2_approx(fmaf(__uint_as_float(su[i]), p.scale_log2, -buf[i]));
            pr[i] = (key_ok && i >= lim) ? e : 0.f;
          }
        }
        bwd_store_p(tS, pr, hilo);
        bwd_store_ds(tD, pr, hilo, [&](int i) { return buf[128 + i]; });
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_P);   // also when dead: the MMA warp's waits stay bounded
    }
    // ---- epilogue: dV and dK rows of the tile (zero past kv_len)
    // (one decision per warp: the TMEM loads below are warp-collective)
    bool have = nsteps > 0 && !dead;
    if (have) have = __all_sync(0xffffffffu, wait_bar(BAR_ACC, 0, wc) && !*s_abort);
    if (have) tc_fence_after();
    const bool write = kj < p.Skv;
    const size_t out_row = ((size_t)(b * p.Hkv + kvh) * p.Skv + (write ? kj : 0)) * 256;
    bwd_store_row<kBF16>(tmem + 256u + lane_off, have, key_ok ? 1.f : 0.f, write,
                         static_cast<uint8_t*>(p.dv) + out_row);
    bwd_store_row<kBF16>(tmem + 384u + lane_off, have, key_ok ? p.scale : 0.f, write,
                         static_cast<uint8_t*>(p.dk) + out_row);
  } else if (warp == 4) {
    // ============================================================ producer
    if (lane == 0 && nsteps > 0) {
      mbar_arrive_expect_tx(BAR_RES, 2 * SM::kTile);
      bwd_load_tile(sbase + SM::kRes0, &p.tm_k, BAR_RES, k0, b * p.Hkv + kvh);
      bwd_load_tile(sbase + SM::kRes1, &p.tm_v, BAR_RES, k0, b * p.Hkv + kvh);
      int n = 0;
      for (; n < nsteps; ++n) {
        const int s = n & 1;
        // (the MMA warp releases a stage only after it saw the stage's copy
        // land: it stops at a wait that gave up, so a stage is never reused
        // with a copy in flight)
        if (!wait_bar(BAR_EMPTY(s), ((n >> 1) & 1) ^ 1, wc)) break;
        const int g = n / nq, qt = qt_lo + n - g * nq;
        const int plane = b * p.Hq + kvh * p.G + g;
        const uint32_t st = sbase + SM::kStage + s * 2 * SM::kTile;
        mbar_arrive_expect_tx(BAR_FULL(s), 2 * SM::kTile);
        bwd_load_tile(st, &p.tm_q, BAR_FULL(s), qt * 128, plane);
        bwd_load_tile(st + SM::kTile, &p.tm_do, BAR_FULL(s), qt * 128, plane);
      }
      // copies in flight land before the shared memory goes away (whether or
      // not a role gave up: one may give up after this point); each of these
      // phases is its barrier's last, so on the normal path they pass at once
      drain_bar(BAR_RES, 0, wc.timeout);
      for (int i = n > 2 ? n - 2 : 0; i < n; ++i) drain_bar(BAR_FULL(i & 1), (i >> 1) & 1, wc.timeout);
    }
    __syncwarp();
  } else {
    // ============================================================ MMA issuer
    const uint32_t lead = elect_lane();
    const uint64_t a_k = sw128_desc(sbase + SM::kRes0, 16, 1024);   // K, K-major (A of S^T)
    const uint64_t a_v = sw128_desc(sbase + SM::kRes1, 16, 1024);   // V, K-major (A of dP^T)
    bool ok = nsteps > 0 && warp_wait(BAR_RES, 0, wc);
#pragma unroll 1
    for (int n = 0; n < nsteps && ok; ++n) {
      const int s = n & 1;
      if (!warp_wait(BAR_FULL(s), (n >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sq = sbase + SM::kStage + s * 2 * SM::kTile, sdo = sq + SM::kTile;
      const uint64_t b_q = sw128_desc(sq, 16, 1024), b_do = sw128_desc(sdo, 16, 1024);
      // S^T = K Q^T and dP^T = V dO^T (issued after the previous step's
      // products, which read P^T / dS^T from these columns)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_if(tmem, a_k + kmajor_step(kk), b_q + kmajor_step(kk), kIdescBwdSS, kk > 0, lead);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_if(tmem + 128u, a_v + kmajor_step(kk), b_do + kmajor_step(kk), kIdescBwdSS, kk > 0,
                  lead);
      mma_commit_if(BAR_S, lead);
      __syncwarp();
      if (!warp_wait(BAR_P, n & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int g = n / nq, qt = qt_lo + n - g * nq;
      (void)g;
      const bool hilo = p.G > 1 || bwd_hilo(qt * 128, kv_len, p.causal);
      const uint64_t m_q = sw128_desc(sq, 128 * 128, 1024), m_do = sw128_desc(sdo, 128 * 128, 1024);
      // dV += P^T dO, dK += dS^T Q (K = the step's 128 queries)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_if(tmem + 256u, tmem + 8u * kk, m_do + mnmajor_step(kk), kIdescBwdTS,
                  (n > 0 || kk > 0) ? 1u : 0u, lead);
      if (hilo) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_if(tmem + 256u, tmem + 64u + 8u * kk, m_do + mnmajor_step(kk), kIdescBwdTS, 1u, lead);
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_if(tmem + 384u, tmem + 128u + 8u * kk, m_q + mnmajor_step(kk), kIdescBwdTS,
                  (n > 0 || kk > 0) ? 1u : 0u, lead);
      if (hilo) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_if(tmem + 384u, tmem + 192u + 8u * kk, m_q + mnmajor_step(kk), kIdescBwdTS, 1u, lead);
      }
      mma_commit_if(BAR_EMPTY(s), lead);
      __syncwarp();
    }
    if (!ok && nsteps > 0) *s_abort = 1;
    mma_commit_if(BAR_ACC, lead);   // every product of the tile (or none) has completed
    if (lead) {
      mma_commit(BAR_DRAIN);
      drain_bar(BAR_DRAIN, 0, wc.timeout);
    }
    __syncwarp();
  }

  bwd_teardown(tmem);
}

// ---------------------------------------------------------------------------
// dQ of one 128-row query tile.  TMEM: S / (unused P) at 0, dP / dS at 128,
// dQ at 256 (rows = queries).
template <bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using SM = BwdSmem;
  extern __shared__ uint8_t smem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heaviest query tiles (the last ones, under a causal mask) first
  const int per_qt = p.B * p.Hq;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / per_qt);
  const int bh = blockIdx.x % per_qt;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int kvh = h / p.G;
  const int q_len = p.seqlens ? min(p.seqlens[b], p.Sq) : p.Sq;
  const int kv_len = p.seqlens ? min(p.seqlens[b], p.Skv) : p.Skv;
  const int q0 = qt * 128;
  const int nsteps = dense_tiles(qt, p.n_qt, q_len, kv_len, p.causal ? 1 : 0);   // key tiles [0, n)

  BwdCta cta;
  const uint32_t tmem = bwd_setup(cta, smem_raw);
  const uint32_t sbase = cta.sbase;
  const uint32_t BAR_RES = cta.res(), BAR_S = cta.s_ready(), BAR_P = cta.p_ready(),
                 BAR_ACC = cta.acc(), BAR_DRAIN = cta.drain();
  auto BAR_FULL = [=](int s) { return cta.full(s); };
  auto BAR_EMPTY = [=](int s) { return cta.empty(s); };
  volatile int* s_abort = cta.s_abort;
  const WaitCtx wc{s_abort, p.status, p.timeout_ns};

  if (warp < 4) {
    // ============================================================ elementwise
    const int row = warp * 32 + lane;   // query row of the tile
    const int qi = q0 + row;
    const bool live = qi < q_len;
    const size_t r = (size_t)(b * p.Hq + h) * p.Sq + (live ? qi : 0);
    const float lse = live ? p.lse[r] : INFINITY;
    const float lse2 = (lse == INFINITY) ? INFINITY : lse * kLog2e;
    const float d = live ? p.d_row[r] : 0.f;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off, tD = tmem + 128u + lane_off;
    const bool hilo = bwd_hilo(q0, kv_len, p.causal);
    bool dead = false;
#pragma unroll 1
    for (int n = 0; n < nsteps; ++n) {
      if (!dead && !__all_sync(0xffffffffu, wait_bar(BAR_S, n & 1, wc))) dead = true;
      if (!dead) {
        tc_fence_after();
        const int kbase = n * 128;
        // key column j is valid iff kbase + j < kv_len and (causal) kbase + j <= qi
        const int lim = min(kv_len - kbase, p.causal ? qi - kbase + 1 : 128);
        float pr[128];
        {
          uint32_t su[128];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            tmem_ld32(tS + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&su[32 * cc]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            const float e = ex2_approx(fmaf(__uint_as_float(su[i]), p.scale_log2, -lse2));
            pr[i] = (i < lim) ? e : 0.f;
          }
        }
        bwd_store_ds(tD, pr, hilo, [&](int) { return d; });
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_P);
    }
    // ---- epilogue: the dQ row (zero past q_len)
    // (one decision per warp: the TMEM loads below are warp-collective)
    bool have = nsteps > 0 && !dead;
    if (have) have = __all_sync(0xffffffffu, wait_bar(BAR_ACC, 0, wc) && !*s_abort);
    if (have) tc_fence_after();
    const bool write = qi < p.Sq;
    bwd_store_row<kBF16>(tmem + 256u + lane_off, have, live ? p.scale : 0.f, write,
                         static_cast<uint8_t*>(p.dq) + ((size_t)(b * p.Hq + h) * p.Sq + (write ? qi : 0)) * 256);
  } else if (warp == 4) {
    // ============================================================ producer
    if (lane == 0 && nsteps > 0) {
      mbar_arrive_expect_tx(BAR_RES, 2 * SM::kTile);
      bwd_load_tile(sbase + SM::kRes0, &p.tm_q, BAR_RES, q0, b * p.Hq + h);
      bwd_load_tile(sbase + SM::kRes1, &p.tm_do, BAR_RES, q0, b * p.Hq + h);
      int n = 0;
      for (; n < nsteps; ++n) {
        const int s = n & 1;
        if (!wait_bar(BAR_EMPTY(s), ((n >> 1) & 1) ^ 1, wc)) break;   // (as in the dK / dV kernel)
        const uint32_t st = sbase + SM::kStage + s * 2 * SM::kTile;
        mbar_arrive_expect_tx(BAR_FULL(s), 2 * SM::kTile);
        bwd_load_tile(st, &p.tm_k, BAR_FULL(s), n * 128, b * p.Hkv + kvh);
        bwd_load_tile(st + SM::kTile, &p.tm_v, BAR_FULL(s), n * 128, b * p.Hkv + kvh);
      }
      drain_bar(BAR_RES, 0, wc.timeout);   // as in the dK / dV kernel
      for (int i = n > 2 ? n - 2 : 0; i < n; ++i) drain_bar(BAR_FULL(i & 1), (i >> 1) & 1, wc.timeout);
    }
    __syncwarp();
  } else {
    // ============================================================ MMA issuer
    const uint32_t lead = elect_lane();
    const uint64_t a_q = sw128_desc(sbase + SM::kRes0, 16, 1024);    // Q, K-major (A of S)
    const uint64_t a_do = sw128_desc(sbase + SM::kRes1, 16, 1024);   // dO, K-major (A of dP)
    const bool hilo = bwd_hilo(q0, kv_len, p.causal);
    bool ok = nsteps > 0 && warp_wait(BAR_RES, 0, wc);
#pragma unroll 1
    for (int n = 0; n < nsteps && ok; ++n) {
      const int s = n & 1;
      if (!warp_wait(BAR_FULL(s), (n >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sk = sbase + SM::kStage + s * 2 * SM::kTile, sv = sk + SM::kTile;
      const uint64_t b_k = sw128_desc(sk, 16, 1024), b_v = sw128_desc(sv, 16, 1024);
      // S = Q K^T, dP = dO V^T
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_if(tmem, a_q + kmajor_step(kk), b_k + kmajor_step(kk), kIdescBwdSS, kk > 0, lead);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_if(tmem + 128u, a_do + kmajor_step(kk), b_v + kmajor_step(kk), kIdescBwdSS, kk > 0,
                  lead);
      mma_commit_if(BAR_S, lead);
      __syncwarp();
      if (!warp_wait(BAR_P, n & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dQ += dS K (K = the step's 128 keys; K read MN-major)
      const uint64_t m_k = sw128_desc(sk, 128 * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_if(tmem + 256u, tmem + 128u + 8u * kk, m_k + mnmajor_step(kk), kIdescBwdTS,
                  (n > 0 || kk > 0) ? 1u : 0u, lead);
      if (hilo) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_if(tmem + 256u, tmem + 192u + 8u * kk, m_k + mnmajor_step(kk), kIdescBwdTS, 1u, lead);
      }
      mma_commit_if(BAR_EMPTY(s), lead);
      __syncwarp();
    }
    if (!ok && nsteps > 0) *s_abort = 1;
    mma_commit_if(BAR_ACC, lead);
    if (lead) {
      mma_commit(BAR_DRAIN);
      drain_bar(BAR_DRAIN, 0, wc.timeout);
    }
    __syncwarp();
  }

  bwd_teardown(tmem);
}

// d_row = rowsum(dO * (O + O_lo)) in fp32, one warp per row of D values
// (D a multiple of 4: each lane takes 4 consecutive values per step).
template <bool kBF16>
__global__ void __launch_bounds__(256) fa_bwd_drow_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ o_lo,
                                                          const uint16_t* __restrict__ dout,
                                                          float* __restrict__ d_row, long long rows,
                                                          int D) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  auto lo = [](uint32_t w) { return kBF16 ? __uint_as_float(w << 16) : f16_lo_to_f32(w); };
  auto hi = [](uint32_t w) { return kBF16 ? __uint_as_float(w & 0xFFFF0000u) : f16_hi_to_f32(w); };
  float acc = 0.f;
  for (int c = 4 * lane; c < D; c += 128) {
    const uint2 vo = *reinterpret_cast<const uint2*>(o + r * D + c);
    const uint2 vd = *reinterpret_cast<const uint2*>(dout + r * D + c);
    const uint2 vl = o_lo ? *reinterpret_cast<const uint2*>(o_lo + r * D + c) : make_uint2(0u, 0u);
    acc = fmaf(lo(vd.x), lo(vo.x) + lo(vl.x), acc);
    acc = fmaf(hi(vd.x), hi(vo.x) + hi(vl.x), acc);
    acc = fmaf(lo(vd.y), lo(vo.y) + lo(vl.y), acc);
    acc = fmaf(hi(vd.y), hi(vo.y) + hi(vl.y), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) d_row[r] = acc;
}

}  // namespace fa
