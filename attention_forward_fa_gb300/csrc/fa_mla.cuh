// Top-k sparse attention over a shared latent (sparse MLA forward) for sm_103a.
//
// Every query token t gathers its own key set, the valid slots of
// topk_idx[b, t, :], shared by all query heads (one latent KV head).  A key row
// is [latent (512) | rope (64)], D = 576, and V is the latent part of the same
// row (Dv = 512): "Sparse-MLA training forward: exact running max vs lazy
// rescale" (cf-1.com), section "Background: sparse MLA and top-k gathered KV".
//
// One CTA per (token, group of 128 query heads, quarter of Dv): the 128 heads
// are the 128 rows of every MMA.  The fp32 O accumulator of all 512 value
// columns would fill the whole TMEM, so each CTA keeps a quarter (128
// columns) and recomputes S = Q K^T for its quarter.  TMEM (512 columns):
//   [0, 128)    O (this CTA's quarter of Dv), fp32
//   [128, 192)  S of the current 64-key tile, fp32
//   [192, 224)  P, fp16 pairs
//   [224, 512)  Q as fp16 pairs, the A operand of S = Q K^T (576 / 2 columns)
// K is read from an fp16 copy of the latent (bf16 inputs are converted once per
// call), so that the same shared-memory tile is the B operand of both
// products: K-major for Q K^T over all 576 columns, MN-major for P V over this
// CTA's 128 value columns.  Tiles of 64 gathered rows are copied in 16-byte
// chunks (cp.async, one producer warp per stage of a three-stage ring; TMA row
// gathers move far fewer bytes per cycle for 128-byte rows); the Q tile is
// first staged (bf16 or fp16, via TMA) in ring stages 0-1 and converted to
// fp16 into TMEM.
//
// Warps: 0-3 Q conversion, softmax (one thread per head row) and epilogue;
// warps 4-6 producers (warp 4 also issues the Q tile's TMA); warp 7 TMEM
// allocator and MMA issuer.
// MMA order: S_0, then per tile j: S_{j+1} = Q K_{j+1}^T, O += P_j V_j, so the
// softmax of tile j overlaps the next Q K^T.  A tile gets a second P.V pass
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
constexpr int kMlaDq = 128;                  // value columns per CTA
constexpr int kMlaSplit = kMlaDv / kMlaDq;   // CTAs per (token, head group)
constexpr int kMlaHeads = 128;               // query heads per CTA (MMA rows)
constexpr int kMlaNS = 3;                    // ring stages
constexpr int kMlaMaxTopk = 2048;            // longest slot list
constexpr int kMlaThreads = 256;
constexpr int kMlaBoxes = kMlaD / 64;        // 128-byte column boxes per key row
constexpr int kMlaHiLoKeys = 256;
constexpr uint32_t kMlaColO = 0, kMlaColS = 128, kMlaColP = 192, kMlaColQ = 224;

struct MlaParams {
  CUtensorMap tm_q;   // 3-D (D, Sq, B*Hq), box 64 x 1 x 128 heads
  const uint16_t* kl; // fp16 key latent [B, Skv, 576]
  void* o;
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
  static constexpr int kStageBytes = kMlaBoxes * kBoxBytes;      // one gathered tile
  static constexpr int kQBoxBytes = kMlaHeads * 128;             // 128 heads x 64 columns
  static constexpr int kRingOff = 0;
  static constexpr int kIdxOff = kRingOff + kMlaNS * kStageBytes;
  static constexpr int kCntOff = kIdxOff + kMlaMaxTopk * 4;
  static constexpr int kBarOff = kCntOff + (kMlaMaxTopk / 128) * 4 * 4;
  // full[NS], empty[NS], q_full, q_done, s_full, s_free, p_ready, pv_done, drain
  static constexpr int kNumBars = 2 * kMlaNS + 7;
  // tmem base, abort flag, key count, residual-pass flags of two tiles
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kMlaBoxes * kQBoxBytes <= 2 * kStageBytes, "Q staging must fit in stages 0-1");
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// Ring position of gathered tile j: the Q tile occupies the first two stages
// at first, so tile 0 goes to stage 2 and tile j to stage (j + 2) % 3.  `use`
// counts the tiles placed in that stage before this one.
__device__ __forceinline__ void mla_stage(int j, int& s, int& use) {
  const int u = j + 2;
  s = u % kMlaNS;
  use = (s == 2) ? u / kMlaNS : u / kMlaNS - 1;
}

template <bool kBF16>
__global__ void __launch_bounds__(kMlaThreads, 1)
    fa_mla_topk_kernel(const __grid_constant__ MlaParams p) {
  using SM = MlaSmem;
  constexpr uint32_t kIdescQK = idesc_f16(kMlaHeads, kMlaN, false, false);   // fp16 Q x fp16 K
  constexpr uint32_t kIdescPV = idesc_f16(kMlaHeads, kMlaDq, false, true);   // fp16 P x fp16 V

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sRing = sbase + SM::kRingOff;
  int* s_idx = reinterpret_cast<int*>(smem + SM::kIdxOff);
  int* s_cnt = reinterpret_cast<int*>(smem + SM::kCntOff);
  const uint32_t bar0 = sbase + SM::kBarOff;
  const uint32_t BAR_QFULL = bar0 + 8u * (2 * kMlaNS);
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
  const int qtr = blockIdx.x % kMlaSplit;
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
      mbar_init(bar0 + 8u * s, 1);              // full: TMA bytes
      mbar_init(bar0 + 8u * (kMlaNS + s), 1);   // empty: MMA commit
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
  if (warp == 7) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();

  // The Q tile (bf16 or fp16) into ring stages 0-1 while the softmax warps
  // compact the key list.
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
      // ---- Q: staging -> fp16 pairs in TMEM columns [224, 512)
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
          tmem_st32(tmem + lane_off + kMlaColQ + 32 * bx, w);
        }
        tmem_wait_st();
        if (kBF16 && row_ok && ((amax & 0xFFFFu) > 0x477Fu || (amax >> 16) > 0x477Fu))
          atomicOr(p.status, kStatusRange);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_QDONE);   // Q in TMEM, staging free

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
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = sv[i];
#pragma unroll
          for (int i = 8; i < kMlaN; i += 16)
#pragma unroll
            for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], sv[i + q], sv[i + 8 + q]);
          const float mb =
              fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
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
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < kMlaDq / 32; ++cc) {
            uint32_t o32[32];
            tmem_ld32(tO + 32 * cc, o32);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o32[2 * i]), __uint_as_float(o32[2 * i + 1])),
                               a2),
                        x0, x1);
              o32[2 * i] = __float_as_uint(x0);
              o32[2 * i + 1] = __float_as_uint(x1);
            }
            tmem_st32(tO + 32 * cc, o32);
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

    // ---- epilogue: O / l for this CTA's 128 value columns, LSE (quarter 0)
    const bool acc = nt > 0 && !dead &&
                     __all_sync(0xffffffffu, wait_bar(BAR_PVDONE, (npv - 1) & 1, wc));
    if (acc) tc_fence_after();
    const bool write = row_ok;
    const float inv_l = (acc && l > 0.f) ? 1.f / l : 0.f;
    uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                     ((size_t)(b * p.Hq + h) * p.Sq + t) * kMlaDv + qtr * kMlaDq;
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
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = __uint_as_float(o32[8 * i + 2 * e]) * inv_l;
            const float a1 = __uint_as_float(o32[8 * i + 2 * e + 1]) * inv_l;
            w[e] = kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
          }
          dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    if (write && qtr == 0)
      p.lse[(size_t)(b * p.Hq + h) * p.Sq + t] =
          (acc && l > 0.f) ? __fmaf_rn(m, p.scale, __logf(l)) : INFINITY;
  } else if (warp < 4 + kMlaNS) {
    // ============================================================ producers
    // Warp 4 + s fills ring stage s: the tiles j with (j + 2) % 3 == s.  Each
    // lane copies 16-byte chunks (4 rows x 128 bytes per warp instruction, so
    // every 128-byte line is read whole) to their 128-byte-swizzle positions,
    // then the warp waits for its copies, fences them for the tensor core (async
    // proxy) and arrives on the stage's full barrier.
    const int s = warp - 4;
    const uint32_t stage = sRing + s * SM::kStageBytes;
    const int sub = lane >> 3;       // row within a group of four
    const int chunk = lane & 7;      // 16-byte chunk within a 128-byte row
    bool ab = false;
#pragma unroll 1
    for (int j = (s + 1) % kMlaNS; j < nt && !ab; j += kMlaNS) {
      int s_, use;
      mla_stage(j, s_, use);
      if (lane == 0) {
        if (use == 0 && s < 2) {
          ab = !wait_bar(BAR_QDONE, 0, wc);                             // Q staging consumed
        } else if (use > 0) {
          ab = !wait_bar(bar0 + 8u * (kMlaNS + s), (use - 1) & 1, wc);   // stage released
        }
      }
      ab = __shfl_sync(0xffffffffu, ab, 0);
      if (ab) break;
#pragma unroll 1
      for (int g = 0; g < kMlaN / 4; ++g) {
        // positions past the last key repeat a valid row (their scores are masked)
        const int row = 4 * g + sub;
        const int pos = j * kMlaN + row;
        const int key = s_idx[pos < nkeys ? pos : nkeys - 1];
        const uint16_t* src = p.kl + ((size_t)b * p.Skv + key) * kMlaD + chunk * 8;
        const uint32_t dst = stage + row * 128 + ((chunk ^ (row & 7)) << 4);
#pragma unroll
        for (int bx = 0; bx < kMlaBoxes; ++bx) cp_async16(dst + bx * SM::kBoxBytes, src + bx * 64);
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * s);
    }
    // the Q tile's copy must land before the CTA's shared memory goes away
    if (s == 0 && lane == 0 && live) drain_bar(BAR_QFULL, 0, wc.timeout);
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
      const uint64_t v_desc0 = sw128_desc(sRing + qtr * 2 * SM::kBoxBytes, SM::kBoxBytes, 1024);
      int c_pready = 0;   // P-ready phases consumed
#pragma unroll 1
      for (int j = 0; j <= nt && ok; ++j) {
        if (j < nt) {
          // S_j = Q K_j^T, once the softmax of tile j-1 has read S
          if (j > 0) ok = __all_sync(0xffffffffu, wait_bar(BAR_SFREE, (j - 1) & 1, wc));
          int s, use;
          mla_stage(j, s, use);
          if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar0 + 8u * s, use & 1, wc));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = k_desc0 + ((uint32_t)(s * SM::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kMlaD / 16; ++kk) {
            const uint32_t off16 = (uint32_t)((kk >> 2) * SM::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ts_if(tmem + kMlaColS, tmem + kMlaColQ + 8 * kk, kd + off16, kIdescQK, kk > 0, lead);
          }
          mma_commit_if(BAR_SFULL, lead);
        }
        if (j == 0) continue;
        // O += P_{j-1} V_{j-1} (this CTA's 128 value columns of the tile), then
        // the residual pass with P_lo when the softmax asked for one
        const int jp = j - 1;
        int s, use;
        mla_stage(jp, s, use);
        const uint64_t vd = v_desc0 + ((uint32_t)(s * SM::kStageBytes) >> 4);
        for (int pass = 0; pass < 2; ++pass) {
          if (!__all_sync(0xffffffffu, wait_bar(BAR_PREADY, c_pready & 1, wc))) {
            ok = false;
            break;
          }
          ++c_pready;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kMlaN / 16; ++kk)
            mma_ts_if(tmem + kMlaColO, tmem + kMlaColP + 8 * kk, vd + ((kk * 2048) >> 4), kIdescPV,
                      (jp > 0 || pass > 0 || kk > 0) ? 1u : 0u, lead);
          mma_commit_if(BAR_PVDONE, lead);
          if (pass == 0 && !s_lo[jp & 1]) break;
        }
        if (!ok) break;
        mma_commit_if(bar0 + 8u * (kMlaNS + s), lead);   // stage free
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
  if (warp == 7) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
