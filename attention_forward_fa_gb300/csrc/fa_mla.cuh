// Top-k sparse attention over a shared latent (sparse MLA forward) for sm_103a.
//
// Every query token t gathers its own key set, the valid slots of
// topk_idx[b, t, :], shared by all query heads (one latent KV head).  A key row
// is [latent (512) | rope (64)], D = 576, and V is the latent part of the same
// row (Dv = 512): "Sparse-MLA training forward: exact running max vs lazy
// rescale" (cf-1.com), section "Background: sparse MLA and top-k gathered KV".
//
// Two CTAs per (token, group of 128 query heads), one per half of Dv: the 128
// heads are the 128 rows of every MMA.  The fp32 O accumulator of all 512
// value columns would fill the whole TMEM, so each CTA keeps half of it and
// computes S = Q K^T itself.  TMEM (512 columns):
//   [0, 256)    O (this CTA's half of Dv), fp32
//   [256, 320)  S of the current 64-key tile, fp32
//   [320, 352)  P, fp16 pairs
//   [352, 512)  query columns 0-319 as fp16 pairs (A operand of Q K^T from TMEM)
// Query columns 320-575 are kept in shared memory as fp16 (A operand of those
// Q K^T steps from shared memory).  K is read from an fp16 copy of the latent
// (bf16 inputs are converted once per call), so that one gathered tile is the
// B operand of both products: K-major for Q K^T over all 576 columns,
// MN-major for P V over this CTA's 256 value columns.
//
// A ring stage holds one tile of 64 gathered rows (nine 64-column boxes).  It
// has two regions with their own full / empty barriers: V, this CTA's four
// value boxes (read by Q K^T and P V), and X, the other five boxes (read by
// Q K^T only).  X is free again once Q K^T of its tile is done, V once its
// P V is done; Q K^T multiplies the X boxes first, and P V of the previous
// tile runs between the two parts, which gives the gather of the V boxes of
// tile j+1 the time of the V steps of tile j and the X steps of tile j+1.  Three producer
// warps copy every tile together in 16-byte chunks (cp.async); the Q tile is
// first staged (bf16 or fp16, via TMA) in both ring stages and converted to
// fp16 into TMEM and shared memory.
//
// Warps: 0-3 Q conversion, softmax (one thread per head row) and epilogue;
// warps 4-6 producers (warp 4 also issues the Q tile's TMA); warp 7 TMEM
// allocator and MMA issuer.
// MMA order per tile j: the X steps of S_j = Q K_j^T, O += P_{j-1} V_{j-1},
// the V steps of S_j; so the softmax of tile j-1 overlaps the X steps of S_j,
// and the V region of tile j-1 is free (for tile j+1) before the V steps of S_j.  A tile gets a second P.V pass
// with the residual P_lo = p - fp16(p) (written over P once the first pass has
// read it) when the token has fewer than kMlaHiLoKeys keys, or when a row keeps
// a stale max below the tile's max (lazy rescale): that row's dominant p is
// then above 1 and not exact in fp16, which peaked rows would show.
#pragma once
#include "fa_tiled.cuh"

namespace fa {

constexpr int kMlaD = 576;                   // key / query width: latent 512 + rope 64
constexpr int kMlaDv = 512;                  // value width (the latent part of a key row)
constexpr int kMlaN = 64;                    // gathered keys per tile
constexpr int kMlaDq = 256;                  // value columns per CTA
constexpr int kMlaSplit = kMlaDv / kMlaDq;   // CTAs per (token, head group)
constexpr int kMlaHeads = 128;               // query heads per CTA (MMA rows)
constexpr int kMlaNS = 2;                    // ring stages
constexpr int kMlaRescaleChunks = 2;         // O columns per TMEM round trip of a rescale: x 32
constexpr int kMlaProducers = 3;             // producer warps, all on every tile
constexpr int kMlaMmaWarp = 4 + kMlaProducers;
constexpr int kMlaThreads = 32 * (kMlaMmaWarp + 1);
constexpr int kMlaMaxTopk = 2048;            // longest slot list
constexpr int kMlaBoxes = kMlaD / 64;        // 128-byte column boxes per key row
constexpr int kMlaQtBoxes = 5;               // query boxes kept in TMEM (columns 0-319)
// Tokens with fewer keys than this take the hi + lo split on every tile.  The
// sparse-MLA rows are peaked (a few keys carry most of the weight), so fp16
// P alone leaves less margin than on the dense kernel's rows: in an fp16-P
// emulation of the kernel, rows of 256-300 keys reach 1.15x the elementwise
// bound, rows of 512 keys and more stay at or below 0.65x.
constexpr int kMlaHiLoKeys = 512;
constexpr uint32_t kMlaColO = 0, kMlaColS = 256, kMlaColP = 320, kMlaColQ = 352;
static_assert(kMlaColQ + 32 * kMlaQtBoxes == 512, "TMEM plan");

struct MlaParams {
  CUtensorMap tm_q;   // 3-D (D, Sq, B*Hq), box 64 x 1 x 128 heads
  const uint16_t* kl; // fp16 key latent [B, Skv, 576]
  void* o;
  void* o_lo;       // optional: o's rounding residual, same type and layout (or null)
  float* lse;
  const int* seqlens;
  const int* topk;
  long long topk_stride_b;
  int W;              // slots per token
  int B, Hq, Sq, Skv;
  int n_hg;           // ceil(Hq / 128)
  int q_rows;         // head rows of the Q box: min(128, B * Hq)
  int causal;         // keys j > t masked
  float scale, scale_log2, threshold;
  long long timeout_ns;
  int* status;
};

struct MlaSmem {
  static constexpr int kBoxBytes = kMlaN * 128;                  // 64 key rows x 64 columns
  static constexpr int kStageBytes = kMlaBoxes * kBoxBytes;      // one gathered tile (72 KB)
  static constexpr int kQBoxBytes = kMlaHeads * 128;             // 128 heads x 64 columns
  static constexpr int kRingOff = 0;
  static constexpr int kQsOff = kRingOff + kMlaNS * kStageBytes;  // query columns 320-575
  static constexpr int kIdxOff = kQsOff + (kMlaBoxes - kMlaQtBoxes) * kQBoxBytes;
  static constexpr int kCntOff = kIdxOff + kMlaMaxTopk * 4;
  static constexpr int kBarOff = kCntOff + (kMlaMaxTopk / 128) * 4 * 4;
  // full_x[NS], full_v[NS], empty_x[NS], empty_v[NS], q_full, q_done, s_full,
  // s_free, p_ready, pv_done, drain
  static constexpr int kNumBars = 4 * kMlaNS + 7;
  // tmem base, abort flag, key count, residual-pass flags of two tiles
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kMlaBoxes * kQBoxBytes <= kMlaNS * kStageBytes, "Q staging must fit in the ring");
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// The V boxes of the CTA for value half `half` are 4 half .. 4 half + 3; every
// other box of a key row is an X box.
__device__ __forceinline__ bool mla_is_v_box(int bx, int half) { return (bx >> 2) == half && bx < 8; }

// Waits until at most one committed group of this thread's cp.async copies
// is pending (the producers keep two regions in flight).
__device__ __forceinline__ void cp_async_wait_one_pending() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// One part of Q K^T for a tile: the steps over the X boxes (kV false, the
// first steps of the product) or over the V boxes (k-step kk covers query
// columns 16 kk .. 16 kk + 15: box kk / 4).  Query columns below 320 come from
// TMEM, the others from shared memory.
template <int kHalf, bool kV>
__device__ __forceinline__ void mla_issue_qk(uint32_t tmem, uint64_t kd, uint64_t qs_desc0,
                                             uint32_t idesc, uint32_t lead) {
  constexpr int kSteps = kMlaD / 16;
  bool first = !kV;
#pragma unroll
  for (int kk = 0; kk < kSteps; ++kk) {
    const bool in_v = ((kk >> 4) == kHalf) && kk < 32;
    if (in_v != kV) continue;
    const uint32_t boff16 = (uint32_t)((kk >> 2) * MlaSmem::kBoxBytes + (kk & 3) * 32) >> 4;
    if (kk < 4 * kMlaQtBoxes) {
      mma_ts_if(tmem + kMlaColS, tmem + kMlaColQ + 8 * kk, kd + boff16, idesc, first ? 0u : 1u,
                lead);
    } else {
      const int qk = kk - 4 * kMlaQtBoxes;
      const uint32_t aoff16 = (uint32_t)((qk >> 2) * MlaSmem::kQBoxBytes + (qk & 3) * 32) >> 4;
      mma_ss_if(tmem + kMlaColS, qs_desc0 + aoff16, kd + boff16, idesc, first ? 0u : 1u, lead);
    }
    first = false;
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kMlaThreads, 1)
    fa_mla_topk_kernel(const __grid_constant__ MlaParams p) {
  using SM = MlaSmem;
  constexpr uint32_t kIdescQK = idesc_f16(kMlaHeads, kMlaN, false, false);   // fp16 Q x fp16 K
  constexpr uint32_t kIdescPV = idesc_f16(kMlaHeads, kMlaDq, false, true);   // fp16 P x fp16 V

  // The next call on the stream may be scheduled once every CTA of this one
  // has started; nothing below touches global memory before the previous
  // kernel (the latent conversion, or the previous call) has completed.
  pdl_launch_dependents();
  pdl_wait_prior();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sRing = sbase + SM::kRingOff;
  const uint32_t sQs = sbase + SM::kQsOff;
  int* s_idx = reinterpret_cast<int*>(smem + SM::kIdxOff);
  int* s_cnt = reinterpret_cast<int*>(smem + SM::kCntOff);
  const uint32_t bar0 = sbase + SM::kBarOff;
  auto BAR_FULL_X = [=](int s) { return bar0 + 8u * s; };
  auto BAR_FULL_V = [=](int s) { return bar0 + 8u * (kMlaNS + s); };
  auto BAR_EMPTY_X = [=](int s) { return bar0 + 8u * (2 * kMlaNS + s); };
  auto BAR_EMPTY_V = [=](int s) { return bar0 + 8u * (3 * kMlaNS + s); };
  const uint32_t BAR_QFULL = bar0 + 8u * (4 * kMlaNS);
  const uint32_t BAR_QDONE = BAR_QFULL + 8;
  const uint32_t BAR_SFULL = BAR_QFULL + 16;
  const uint32_t BAR_SFREE = BAR_QFULL + 24;
  const uint32_t BAR_PREADY = BAR_QFULL + 32;
  const uint32_t BAR_PVDONE = BAR_QFULL + 40;
  const uint32_t BAR_DRAIN = BAR_QFULL + 48;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SM::kMiscOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + SM::kMiscOff + 4);
  int* s_nkeys = reinterpret_cast<int*>(smem + SM::kMiscOff + 8);
  volatile int* s_lo = reinterpret_cast<volatile int*>(smem + SM::kMiscOff + 12);   // [2]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---------------------------------------------------------------- unit
  const int half = blockIdx.x % kMlaSplit;
  const int rest = blockIdx.x / kMlaSplit;
  const int hg = rest % p.n_hg;
  const int bt = rest / p.n_hg;
  const int b = bt / p.Sq;
  const int t = p.Sq - 1 - bt % p.Sq;   // later tokens (longer key lists) first
  const int q_len = p.seqlens ? min(p.seqlens[b], p.Sq) : p.Sq;
  const int kv_len = p.seqlens ? min(p.seqlens[b], p.Skv) : p.Skv;
  const bool live = t < q_len && kv_len > 0;

  if (tid == 0) {
    for (int s = 0; s < kMlaNS; ++s) {
      mbar_init(BAR_FULL_X(s), kMlaProducers);   // one arrival per producer warp
      mbar_init(BAR_FULL_V(s), kMlaProducers);
      mbar_init(BAR_EMPTY_X(s), 1);              // MMA commits
      mbar_init(BAR_EMPTY_V(s), 1);
    }
    mbar_init(BAR_QFULL, 1);
    mbar_init(BAR_QDONE, 4);     // one arrival per softmax warp
    mbar_init(BAR_SFULL, 1);
    mbar_init(BAR_SFREE, 4);
    mbar_init(BAR_PREADY, 4);
    mbar_init(BAR_PVDONE, 1);
    mbar_init(BAR_DRAIN, 1);
    *s_abort = 0;
    *s_nkeys = 0;
    fence_mbar_init();
  }
  if (warp == kMlaMmaWarp) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();

  // The Q tile (bf16 or fp16) into the ring while the softmax warps compact
  // the key list.
  if (warp == 4 && lane == 0 && live) {
    tma_prefetch_desc(&p.tm_q);
    mbar_arrive_expect_tx(BAR_QFULL, kMlaBoxes * 128 * p.q_rows);
    for (int bx = 0; bx < kMlaBoxes; ++bx)
      tma_load_3d(sRing + bx * SM::kQBoxBytes, &p.tm_q, BAR_QFULL, 64 * bx, t,
                  b * p.Hq + hg * kMlaHeads);
  }
  // Valid slots of this token, in slot order: 0 <= idx < kv_len and, with the
  // causal flag, idx <= t.  A key listed by two slots is kept twice.
  if (warp < 4 && live) {
    const int* row = p.topk + (long long)b * p.topk_stride_b + (long long)t * p.W;
    constexpr int kRounds = kMlaMaxTopk / 128;
    int v[kRounds];
#pragma unroll
    for (int i = 0; i < kRounds; ++i) {
      const int s = i * 128 + tid;
      v[i] = (s < p.W) ? __ldg(row + s) : -1;
    }
    unsigned bal[kRounds];
#pragma unroll
    for (int i = 0; i < kRounds; ++i) {
      const bool ok = v[i] >= 0 && v[i] < kv_len && (!p.causal || v[i] <= t);
      bal[i] = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) s_cnt[i * 4 + warp] = __popc(bal[i]);
    }
    named_sync(1, 128);
    int total = 0;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kRounds; ++i) {
      const int c0 = s_cnt[i * 4], c1 = s_cnt[i * 4 + 1], c2 = s_cnt[i * 4 + 2],
                c3 = s_cnt[i * 4 + 3];
      const int before = (warp > 0 ? c0 : 0) + (warp > 1 ? c1 : 0) + (warp > 2 ? c2 : 0);
      if ((bal[i] >> lane) & 1u) s_idx[total + before + __popc(bal[i] & lt)] = v[i];
      total += c0 + c1 + c2 + c3;
    }
    if (tid == 0) *s_nkeys = total;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int nkeys = *s_nkeys;
  const int nt = (nkeys + kMlaN - 1) / kMlaN;
  const bool hilo = nkeys < kMlaHiLoKeys;
  const WaitCtx wc{s_abort, p.status, p.timeout_ns};

  if (warp < 4) {
    // ============================================================ softmax
    const int r = tid;                       // head row within the group = TMEM lane
    const int h = hg * kMlaHeads + r;
    const bool row_ok = h < p.Hq;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + kMlaColS;
    const uint32_t tP = tmem + lane_off + kMlaColP;
    const uint32_t tO = tmem + lane_off + kMlaColO;
    bool dead = false;
    float m = -INFINITY, l = 0.f;
    int npv = 0;   // P.V passes of the tiles done so far (the MMA warp counts the same)
    if (nt > 0) {
      // ---- Q: staging -> fp16; columns 0-319 as pairs into TMEM columns
      // [352, 512), columns 320-575 into shared memory (same swizzled layout)
      if (!__all_sync(0xffffffffu, wait_bar(BAR_QFULL, 0, wc))) dead = true;
      if (!dead) {
        uint32_t amax = 0;
#pragma unroll 1
        for (int bx = 0; bx < kMlaBoxes; ++bx) {
          const uint8_t* rowp = smem + SM::kRingOff + bx * SM::kQBoxBytes + r * 128;
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(rowp + ((c ^ (r & 7)) << 4));
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (kBF16) {
                amax = max_u16x2(amax, xs[e] & 0x7FFF7FFFu);
                w[4 * c + e] = pack_f16x2(__uint_as_float(xs[e] << 16),
                                          __uint_as_float(xs[e] & 0xFFFF0000u));
              } else {
                w[4 * c + e] = xs[e];
              }
            }
          }
          if (bx < kMlaQtBoxes) {
            tmem_st32(tmem + lane_off + kMlaColQ + 32 * bx, w);
          } else {
            uint8_t* dst = smem + SM::kQsOff + (bx - kMlaQtBoxes) * SM::kQBoxBytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();   // generic-proxy writes -> tensor core reads
        if (kBF16 && row_ok && ((amax & 0xFFFFu) > 0x477Fu || (amax >> 16) > 0x477Fu))
          atomicOr(p.status, kStatusRange);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_QDONE);   // Q in TMEM / shared memory, staging free

      const float c = p.scale_log2;
      const uint64_t c2 = f2_pack(c, c);
#pragma unroll 1
      for (int j = 0; j < nt; ++j) {
        // Every softmax thread reaches the barrier reduction once per tile, also
        // after a bounded wait gave up, so that no thread waits on it forever.
        if (!dead && !__all_sync(0xffffffffu, wait_bar(BAR_SFULL, j & 1, wc))) dead = true;
        uint32_t ph[32], pl[32];
        float sv[kMlaN];
        float alpha = 1.f, neg = 0.f;
        bool lo_row = false;
        if (!dead) {
          tc_fence_after();
          uint32_t su[kMlaN];
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&su[0]));
          tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&su[32]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR_SFREE);   // S may be overwritten by the next Q K^T
#pragma unroll
          for (int i = 0; i < kMlaN; ++i) sv[i] = __uint_as_float(su[i]);
          const int lim = nkeys - j * kMlaN;   // columns >= lim hold no key
          if (lim < kMlaN) {
#pragma unroll
            for (int i = 0; i < kMlaN; ++i)
              if (i >= lim) sv[i] = -INFINITY;
          }
          const float mb = row_max(sv);
          const float m_new = fmaxf(m, mb);
          float m_use = m_new;
          if (m != -INFINITY) {
            const float step = (m - m_new) * c;   // <= 0, log2 units of scaled scores
            if (step >= -p.threshold) {
              m_use = m;                          // keep the (possibly stale) max
            } else {
              alpha = ex2_approx(step);
            }
          }
          // p > 1 (a kept max below the block max) or a short row: this tile
          // also gets the residual pass P_lo = p - fp16(p)
          lo_row = hilo || mb > m_use;
          neg = (m_use == -INFINITY) ? 0.f : -m_use * c;
          m = m_use;
        }
        // residual pass for the whole CTA? (every softmax thread, once per tile)
        const bool lo = named_or(2, kMlaHeads, lo_row);
        if (!dead) {
          const uint64_t neg2 = f2_pack(neg, neg);
          uint64_t sum2[2] = {0ull, 0ull};
          // (two copies of the loop: the residual test inside it would cost
          // more instructions than the exponentials)
          if (!lo) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float a0, a1;
              f2_unpack(f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), c2, neg2), a0, a1);
              a0 = ex2_approx(a0);
              a1 = ex2_approx(a1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(a0, a1));
              ph[i] = pack_f16x2(a0, a1);
            }
          } else {
            // rows that do not need the residual contribute zeros to its pass
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float a0, a1;
              f2_unpack(f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), c2, neg2), a0, a1);
              a0 = ex2_approx(a0);
              a1 = ex2_approx(a1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(a0, a1));
              ph[i] = pack_f16x2(a0, a1);
              pl[i] = lo_row ? pack_f16x2(a0 - f16_lo_to_f32(ph[i]), a1 - f16_hi_to_f32(ph[i])) : 0u;
            }
          }
          float r0, r1, r2, r3;
          f2_unpack(sum2[0], r0, r1);
          f2_unpack(sum2[1], r2, r3);
          l = __fmaf_rn(alpha, l, (r0 + r1) + (r2 + r3));   // (one rounding in every build)
        }
        if (dead) continue;
        // the previous tile's P.V passes have read P and written O
        if (j > 0 && !__all_sync(0xffffffffu, wait_bar(BAR_PVDONE, (npv - 1) & 1, wc))) {
          dead = true;
          continue;
        }
        tc_fence_after();
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O *= alpha, kMlaRescaleChunks 32-column chunks per TMEM round trip
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int cc = 0; cc < kMlaDq / 32; cc += kMlaRescaleChunks) {
            uint32_t o32[kMlaRescaleChunks][32];
#pragma unroll
            for (int u = 0; u < kMlaRescaleChunks; ++u) tmem_ld32(tO + 32 * (cc + u), o32[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kMlaRescaleChunks; ++u) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float x0, x1;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(o32[u][2 * i]),
                                         __uint_as_float(o32[u][2 * i + 1])),
                                 a2),
                          x0, x1);
                o32[u][2 * i] = __float_as_uint(x0);
                o32[u][2 * i + 1] = __float_as_uint(x1);
              }
              tmem_st32(tO + 32 * (cc + u), o32[u]);
            }
          }
        }
        tmem_st32(tP, ph);
        tmem_wait_st();
        tc_fence_before();
        if (tid == 0) s_lo[j & 1] = lo ? 1 : 0;   // read by the MMA warp after P ready
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_PREADY);
        if (lo) {
          // P_lo replaces P once the first pass of this tile has read it
          if (!__all_sync(0xffffffffu, wait_bar(BAR_PVDONE, npv & 1, wc))) {
            dead = true;
            continue;
          }
          tc_fence_after();
          tmem_st32(tP, pl);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR_PREADY);
        }
        npv += lo ? 2 : 1;
      }
    }

    // ---- epilogue: O / l for this CTA's 256 value columns, LSE (first half)
    const bool acc = nt > 0 && !dead &&
                     __all_sync(0xffffffffu, wait_bar(BAR_PVDONE, (npv - 1) & 1, wc));
    if (acc) tc_fence_after();
    const bool write = row_ok;
    const float inv_l = (acc && l > 0.f) ? 1.f / l : 0.f;
    uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                     ((size_t)(b * p.Hq + h) * p.Sq + t) * kMlaDv + half * kMlaDq;
#pragma unroll 1
    for (int cc = 0; cc < kMlaDq / 32; ++cc) {
      uint32_t o32[32];
      if (acc) {
        tmem_ld32(tO + 32 * cc, o32);   // warp-collective
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o32[i] = 0;
      }
      if (write) {
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
        uint4* dst_lo = p.o_lo ? reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o_lo) +
                                                          (orow - static_cast<uint16_t*>(p.o)) + 32 * cc)
                               : nullptr;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t w[4], wl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = __uint_as_float(o32[8 * i + 2 * e]) * inv_l;
            const float a1 = __uint_as_float(o32[8 * i + 2 * e + 1]) * inv_l;
            w[e] = kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
            wl[e] = pack_residual_x2(a0, a1, w[e], kBF16);
          }
          dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          if (dst_lo) dst_lo[i] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      }
    }
    if (write && half == 0)
      p.lse[(size_t)(b * p.Hq + h) * p.Sq + t] =
          (acc && l > 0.f) ? __fmaf_rn(m, p.scale, __logf(l)) : INFINITY;
  } else if (warp < kMlaMmaWarp) {
    // ============================================================ producers
    // All three warps copy every tile j into stage j % 2: warp 4 + w the row
    // groups w, w + 3, w + 6, ... (four rows each).  A tile is two regions,
    // taken in order: its X boxes, once Q K^T of the tile two back has read
    // them, then its V boxes, once its P.V has.  Each lane copies 16-byte
    // chunks (4 rows x 128 bytes per warp instruction, so every 128-byte line
    // is read whole) to their 128-byte-swizzle positions, one commit group per
    // region.  Two regions are in flight: after issuing region r the warp
    // waits for region r - 1's group only, fences it for the tensor core
    // (async proxy) and arrives on its full barrier.  (Region r's empty
    // barrier never waits on region r - 1's full one: X of tile j frees with
    // Q K^T of tile j - 2 and V with P.V of tile j - 2, both issued before
    // tile j is needed.)  The first use of each stage waits for the Q staging
    // instead.
    const int w = warp - 4;
    const int sub = lane >> 3;       // row within a group of four
    const int chunk = lane & 7;      // 16-byte chunk within a 128-byte row
    bool ab = false;
    auto full_bar = [&](int r) { return (r & 1) ? BAR_FULL_V((r >> 1) % kMlaNS) : BAR_FULL_X((r >> 1) % kMlaNS); };
    int r = 0;
#pragma unroll 1
    for (; r < 2 * nt; ++r) {
      const int j = r >> 1, region = r & 1;
      const int s = j % kMlaNS, use = j / kMlaNS;
      const uint32_t stage = sRing + s * SM::kStageBytes;
      if (lane == 0) {
        if (use == 0) {
          ab = region == 0 && !wait_bar(BAR_QDONE, 0, wc);               // Q staging consumed
        } else {
          ab = !wait_bar(region ? BAR_EMPTY_V(s) : BAR_EMPTY_X(s), (use - 1) & 1, wc);
        }
      }
      ab = __shfl_sync(0xffffffffu, ab, 0);
      if (ab) break;
#pragma unroll 1
      for (int g = w; g < kMlaN / 4; g += kMlaProducers) {
        // positions past the last key repeat a valid row (their scores are masked)
        const int row = 4 * g + sub;
        const int pos = j * kMlaN + row;
        const int key = s_idx[pos < nkeys ? pos : nkeys - 1];
        const uint16_t* src = p.kl + ((size_t)b * p.Skv + key) * kMlaD + chunk * 8;
        const uint32_t dst = stage + row * 128 + ((chunk ^ (row & 7)) << 4);
#pragma unroll
        for (int bx = 0; bx < kMlaBoxes; ++bx)
          if (mla_is_v_box(bx, half) == (region == 1))
            cp_async16(dst + bx * SM::kBoxBytes, src + bx * 64);
      }
      cp_async_commit();
      if (r > 0) {
        cp_async_wait_one_pending();   // region r - 1 landed
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full_bar(r - 1));
      }
    }
    // the last region issued (or, after an abort, every copy in flight)
    cp_async_wait_all();
    if (!ab && r > 0) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(r - 1));
    }
    // the Q tile's copy must land before the CTA's shared memory goes away
    if (w == 0 && lane == 0 && live) drain_bar(BAR_QFULL, 0, wc.timeout);
    __syncwarp();
  } else {
    // ============================================================ MMA issue
    // The whole warp waits and runs the issue code (warp-uniform control flow);
    // only the elected lane's tcgen05 instructions take effect, always the same
    // lane since a commit tracks the MMAs of the thread that issues it.
    if (nt > 0) {
      const uint32_t lead = elect_lane();
      bool ok = __all_sync(0xffffffffu, wait_bar(BAR_QDONE, 0, wc));
      tc_fence_after();
      const uint64_t k_desc0 = sw128_desc(sRing, 16, 1024);                          // K-major
      const uint64_t qs_desc0 = sw128_desc(sQs, 16, 1024);                           // K-major
      const uint64_t v_desc0 =
          sw128_desc(sRing + half * 4 * SM::kBoxBytes, SM::kBoxBytes, 1024);         // MN-major
      int c_pready = 0;   // P-ready phases consumed
#pragma unroll 1
      for (int j = 0; j <= nt && ok; ++j) {
        // Per tile j: the X steps of S_j = Q K_j^T, then O += P_{j-1} V_{j-1}
        // (which frees the V region of stage (j-1) % 2 for tile j+1 early),
        // then the V steps of S_j.
        const int s = j % kMlaNS, use = j / kMlaNS;
        const uint64_t kd = k_desc0 + ((uint32_t)(s * SM::kStageBytes) >> 4);
        if (j < nt) {
          // once the softmax of tile j-1 has read S
          if (j > 0) ok = __all_sync(0xffffffffu, wait_bar(BAR_SFREE, (j - 1) & 1, wc));
          if (ok) ok = __all_sync(0xffffffffu, wait_bar(BAR_FULL_X(s), use & 1, wc));
          if (!ok) break;
          tc_fence_after();
          if (half) mla_issue_qk<1, false>(tmem, kd, qs_desc0, kIdescQK, lead);
          else      mla_issue_qk<0, false>(tmem, kd, qs_desc0, kIdescQK, lead);
        }
        if (j > 0) {
          // O += P_{j-1} V_{j-1} (this CTA's 256 value columns of the tile), then
          // the residual pass with P_lo when the softmax asked for one
          const int jp = j - 1;
          const int sp = jp % kMlaNS;
          const uint64_t vd = v_desc0 + ((uint32_t)(sp * SM::kStageBytes) >> 4);
          for (int pass = 0; pass < 2; ++pass) {
            if (!__all_sync(0xffffffffu, wait_bar(BAR_PREADY, c_pready & 1, wc))) {
              ok = false;
              break;
            }
            ++c_pready;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kMlaN / 16; ++kk)
              mma_ts_if(tmem + kMlaColO, tmem + kMlaColP + 8 * kk, vd + ((kk * 2048) >> 4),
                        kIdescPV, (jp > 0 || pass > 0 || kk > 0) ? 1u : 0u, lead);
            mma_commit_if(BAR_PVDONE, lead);
            if (pass == 0 && !s_lo[jp & 1]) break;
          }
          if (!ok) break;
          mma_commit_if(BAR_EMPTY_V(sp), lead);   // the V boxes of tile j-1 are free again
        }
        if (j < nt) {
          ok = __all_sync(0xffffffffu, wait_bar(BAR_FULL_V(s), use & 1, wc));
          if (!ok) break;
          tc_fence_after();
          if (half) mla_issue_qk<1, true>(tmem, kd, qs_desc0, kIdescQK, lead);
          else      mla_issue_qk<0, true>(tmem, kd, qs_desc0, kIdescQK, lead);
          mma_commit_if(BAR_SFULL, lead);
          mma_commit_if(BAR_EMPTY_X(s), lead);   // the X boxes are read by Q K^T only
        }
      }
      // every MMA has finished before TMEM is released
      if (lead) {
        mma_commit(BAR_DRAIN);
        drain_bar(BAR_DRAIN, 0, wc.timeout);
      }
      __syncwarp();
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMlaMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
