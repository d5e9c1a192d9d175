// Tiled FlashAttention forward for sm_103a: dense, causal, ragged (per-batch
// lengths), GQA and block-sparse (compact KV-block lists), D = Dv in {64, 128}.
//
// One CTA owns up to two 128-row query tiles ("slots") that are processed in
// ping-pong so that the softmax of one overlaps the tensor-core work of the
// other.  Work split inside the CTA (384 threads):
//   warps 0-3   softmax + epilogue of slot 0 (one thread per query row)
//   warps 4-7   softmax + epilogue of slot 1
//   warp  8     TMA producer: Q tiles, then K / V tiles into a ring of stages
//   warp  9     TMEM allocator and tcgen05.mma issuer
//   warps 10-11 bf16 -> fp16 conversion of V tiles in shared memory (bf16 I/O)
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
#include "fa_ptx.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per KV tile
constexpr int kTiledThreads = 384;
constexpr int kMaxSel = 512;      // longest block list a CTA stages in smem
constexpr int kHiLoKeys = 256;    // rows with fewer valid keys use the hi+lo P split

enum : int { kStatusTimeout = 1, kStatusRange = 2 };

struct TiledParams {
  CUtensorMap tm_q, tm_k, tm_v;
  void* o;
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
  float scale, scale_log2, threshold;
  long long timeout_ns;
  int* status;
};

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <int D, int NS>
struct TiledSmem {
  static constexpr int kQBytes = kBM * D * 2;           // one query tile
  static constexpr int kStageBytes = kBN * D * 2;       // one K or V tile (Dv == D)
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = 2 * kQBytes;
  static constexpr int kListOff = kStageOff + NS * kStageBytes;
  static constexpr int kBarOff = kListOff + 2 * kMaxSel * 4;
  // barriers: q_full[2], full[NS], empty[NS], vready[NS], s_full[2], p_full[2],
  // o_ready[2], drain
  static constexpr int kNumBars = 2 + 3 * NS + 6 + 1;
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
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (*c.abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if ((long long)(globaltimer_ns() - t0) > c.timeout) {
      *c.abort = 1;
      atomicOr(c.status, kStatusTimeout);
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag (teardown: let copies in flight land).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, long long timeout) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > timeout) return;
  }
}

// The order in which the MMA warp consumes K / V tiles.  f(is_pv, slot, j,
// load, release) is called per MMA group; `load` marks the first use of a
// tile (a new ring stage), `release` the last.  With `shared`, slot 1 reads the
// tiles slot 0 loaded (same KV head and KV tile sequence, n0 <= n1).
template <class F>
__device__ __forceinline__ void for_each_event(int n0, int n1, bool shared, F&& f) {
  auto ev = [&](bool pv, int t, int j) -> bool {
    const int nt = t ? n1 : n0;
    if (j >= nt) return true;
    const bool load = shared ? (t == 0 || j >= n0) : true;
    const bool rel = shared ? (t == 1) : true;
    return f(pv, t, j, load, rel);
  };
  if (!ev(false, 0, 0)) return;
  if (!ev(false, 1, 0)) return;
  const int n = n0 > n1 ? n0 : n1;
  for (int j = 0; j < n; ++j) {
    if (!ev(true, 0, j)) return;
    if (!ev(false, 0, j + 1)) return;
    if (!ev(true, 1, j)) return;
    if (!ev(false, 1, j + 1)) return;
  }
}

template <int D, bool kBF16, int NS>
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
  auto BAR_QFULL = [&](int t) { return bar0 + 8u * t; };
  auto BAR_FULL = [&](int s) { return bar0 + 8u * (2 + s); };
  auto BAR_EMPTY = [&](int s) { return bar0 + 8u * (2 + NS + s); };
  auto BAR_VREADY = [&](int s) { return bar0 + 8u * (2 + 2 * NS + s); };
  auto BAR_SFULL = [&](int t) { return bar0 + 8u * (2 + 3 * NS + t); };
  auto BAR_PFULL = [&](int t) { return bar0 + 8u * (4 + 3 * NS + t); };
  auto BAR_OREADY = [&](int t) { return bar0 + 8u * (6 + 3 * NS + t); };
  const uint32_t BAR_DRAIN = bar0 + 8u * (8 + 3 * NS);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SM::kMiscOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + SM::kMiscOff + 4);
  int* s_slot = reinterpret_cast<int*>(smem + SM::kMiscOff + 8);   // [2] n, [2] hilo

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---------------------------------------------------------------- unit
  const int u = blockIdx.x;
  const int qpos = p.n_qpos - 1 - u / p.units_per_q;   // heaviest query positions first
  const int bh = u % p.units_per_q;
  int b, h_s[2], qt_s[2];
  if (p.pair_mode == 0) {
    b = bh / p.Hq;
    h_s[0] = h_s[1] = bh % p.Hq;
    qt_s[0] = 2 * qpos;
    qt_s[1] = 2 * qpos + 1;
  } else {
    const int hpairs = p.Hq / 2;
    b = bh / hpairs;
    h_s[0] = 2 * (bh % hpairs);
    h_s[1] = h_s[0] + 1;
    qt_s[0] = qt_s[1] = qpos;
  }
  const int kvh = h_s[0] / p.G;   // both slots share it (GQA pairs never straddle a group)
  const int q_len = p.seqlens ? min(p.seqlens[b], p.Sq) : p.Sq;
  const int kv_len = p.seqlens ? min(p.seqlens[b], p.Skv) : p.Skv;
  const int nkb = (p.Skv + kBN - 1) / kBN;
  const bool sparse = p.blk_idx != nullptr;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR_QFULL(t), 1);
      mbar_init(BAR_SFULL(t), 1);
      mbar_init(BAR_PFULL(t), kBM);      // every softmax thread of the slot arrives
      mbar_init(BAR_OREADY(t), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(BAR_FULL(s), 1);
      mbar_init(BAR_EMPTY(s), 1);
      mbar_init(BAR_VREADY(s), 64);     // every converter thread arrives
    }
    mbar_init(BAR_DRAIN, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  // Per-slot KV tile lists and counts.  Dense: the count follows from the
  // lengths and the causal bound.  Block-sparse: warp t compacts the valid
  // slots of its query block (order kept) into s_list[t].
  if (warp < 2) {
    const int t = warp;
    const int qt = qt_s[t];
    const int q0 = qt * kBM;
    int n = 0, hilo = 0;
    const bool live = qt < p.n_qt && q0 < q_len && kv_len > 0;
    if (live && !sparse) {
      int nkv = (kv_len + kBN - 1) / kBN;
      if (p.mask == 1) {
        const int q_last = min(q0 + kBM - 1, q_len - 1);
        nkv = min(nkv, q_last / kBN + 1);
      }
      n = nkv;
      const int min_keys = (p.mask == 1) ? min(q0 + 1, kv_len) : kv_len;
      hilo = min_keys < kHiLoKeys;
    } else if (live && sparse) {
      const int* lst = p.blk_idx + (long long)b * p.blk_stride_b +
                       (long long)h_s[t] * p.blk_stride_h + (long long)qt * p.max_sel;
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
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int n0 = s_slot[0], n1 = s_slot[1];
  const bool shared_kv = !sparse ? (n0 >= 1 && n0 <= n1) : false;
  const WaitCtx wc{s_abort, p.status, p.timeout_ns};
  auto kv_tile = [&](int t, int j) -> int { return sparse ? s_list[t * kMaxSel + j] : j; };

  if (warp == 8) {
    // ============================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      for (int t = 0; t < 2; ++t) {
        if ((t ? n1 : n0) == 0) continue;
        mbar_arrive_expect_tx(BAR_QFULL(t), SM::kQBytes);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sQ + t * SM::kQBytes + bx * (kBM * 128), &p.tm_q, BAR_QFULL(t), 64 * bx,
                      qt_s[t] * kBM, b * p.Hq + h_s[t]);
      }
      int ld = 0;
      for_each_event(n0, n1, shared_kv, [&](bool pv, int t, int j, bool load, bool) -> bool {
        if (!load) return true;
        const int s = ld % NS;
        const uint32_t f = ld / NS;
        ++ld;
        if (!wait_bar(BAR_EMPTY(s), (f & 1) ^ 1, wc)) return false;
        const int kvt = kv_tile(t, j);
        mbar_arrive_expect_tx(BAR_FULL(s), SM::kStageBytes);
        const CUtensorMap* tm = pv ? &p.tm_v : &p.tm_k;
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sStage + s * SM::kStageBytes + bx * (kBN * 128), tm, BAR_FULL(s), 64 * bx,
                      kvt * kBN, b * p.Hkv + kvh);
        return true;
      });
      if (*s_abort) {
        // let every copy in flight land before the CTA's shared memory goes away
        for (int i = (ld > NS ? ld - NS : 0); i < ld; ++i)
          drain_bar(BAR_FULL(i % NS), (i / NS) & 1, wc.timeout);
        for (int t = 0; t < 2; ++t)
          if ((t ? n1 : n0) > 0) drain_bar(BAR_QFULL(t), 0, wc.timeout);
      }
    }
  } else if (warp == 9) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      int ld = 0, vc = 0;
      uint32_t stK = 0, stV = 0;
      const int hilo0 = s_slot[2], hilo1 = s_slot[3];
      for_each_event(n0, n1, shared_kv, [&](bool pv, int t, int j, bool load, bool rel) -> bool {
        uint32_t s;
        if (load) {
          s = ld % NS;
          const uint32_t f = ld / NS;
          ++ld;
          if (pv && kBF16) {
            if (!wait_bar(BAR_VREADY(vc % NS), (vc / NS) & 1, wc)) return false;
            ++vc;
          } else {
            if (!wait_bar(BAR_FULL(s), f & 1, wc)) return false;
          }
          if (pv) stV = s; else stK = s;
        } else {
          s = pv ? stV : stK;
        }
        const uint32_t tS = tmem + 128u * t;
        const uint32_t tO = tmem + 256u + 128u * t;
        if (!pv) {
          if (j == 0 && !wait_bar(BAR_QFULL(t), 0, wc)) return false;
          tc_fence_after();
          const uint32_t qa = sQ + t * SM::kQBytes;
          const uint32_t ka = sStage + s * SM::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kKSteps; ++kk) {
            const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
            mma_ss(tS, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024), kIdescQK,
                   kk > 0);
          }
          mma_commit(BAR_SFULL(t));
        } else {
          if (!wait_bar(BAR_PFULL(t), j & 1, wc)) return false;
          tc_fence_after();
          const uint32_t va = sStage + s * SM::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tO, tS + 8 * kk, sw128_desc(va + kk * 2048, kBN * 128, 1024), kIdescPV,
                   (j > 0 || kk > 0) ? 1u : 0u);
          if (t ? hilo1 : hilo0) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts(tO, tS + 64 + 8 * kk, sw128_desc(va + kk * 2048, kBN * 128, 1024), kIdescPV,
                     1u);
          }
          mma_commit(BAR_OREADY(t));
        }
        if (rel) mma_commit(BAR_EMPTY(s));
        return true;
      });
      // every MMA has finished before TMEM is released
      if (n0 + n1 > 0) {
        mma_commit(BAR_DRAIN);
        drain_bar(BAR_DRAIN, 0, wc.timeout);
      }
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ============================================================ V converter
    if (kBF16) {
      const int ct = tid - 320;   // 0..63
      int ld = 0, vc = 0;
      float amax = 0.f;
      for_each_event(n0, n1, shared_kv, [&](bool pv, int, int, bool load, bool) -> bool {
        if (!load) return true;
        const int s = ld % NS;
        const uint32_t f = ld / NS;
        ++ld;
        if (!pv) return true;
        if (!wait_bar(BAR_FULL(s), f & 1, wc)) return false;
        uint4* base = reinterpret_cast<uint4*>(smem + SM::kStageOff + s * SM::kStageBytes);
#pragma unroll 4
        for (int i = ct; i < SM::kStageBytes / 16; i += 64) {
          uint4 w = base[i];
          uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(ww[e] << 16);
            const float hi = __uint_as_float(ww[e] & 0xFFFF0000u);
            amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
            ww[e] = pack_f16x2(lo, hi);
          }
          base[i] = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(BAR_VREADY(vc % NS));
        ++vc;
        return true;
      });
      if (amax > 65504.f) atomicOr(p.status, kStatusRange);
    }
  } else {
    // ============================================================ softmax + epilogue
    const int t = warp >> 2;
    const int nt = t ? n1 : n0;
    const int hilo = s_slot[2 + t];
    const int qt = qt_s[t];
    const int h = h_s[t];
    const int row = (warp & 3) * 32 + lane;
    const int q0 = qt * kBM;
    const int qi = q0 + row;
    const bool row_valid = qi < q_len;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128u * t + lane_off;
    const uint32_t tO = tmem + 256u + 128u * t + lane_off;
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;   // warp-uniform
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, wait_bar(BAR_SFULL(t), j & 1, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t su[kBN];
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc)
        tmem_ld32(tS + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&su[32 * cc]));
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(su[i]);
      const int kvt = kv_tile(t, j);
      const int kbase = kvt * kBN;
      const bool causal_here = (p.mask == 1) || (p.mask == 2 && kvt == qt);
      const bool need_mask =
          !row_valid || kbase + kBN > kv_len || (causal_here && kbase + kBN - 1 > q0);
      if (need_mask) {
        const int lim_kv = kv_len - kbase;                        // keys >= lim_kv masked
        const int lim_c = causal_here ? qi - kbase + 1 : kBN;     // keys >= lim_c masked
        const int lim = row_valid ? min(lim_kv, lim_c) : 0;
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
      for (int i = 8; i < kBN; ++i) mx[i & 7] = fmaxf(mx[i & 7], s[i]);
      const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
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
      float sm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sm[i] = 0.f;
#pragma unroll
      for (int i = 0; i < kBN; ++i) {
        s[i] = ex2_approx(fmaf(s[i], c, neg));
        sm[i & 7] += s[i];
      }
      const float rs = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
      l = alpha * l + rs;
      m = m_use;
      // rescale O_t; the previous P.V product into O_t must have landed first
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = __all_sync(0xffffffffu, wait_bar(BAR_OREADY(t), (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < Dv / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * cc, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + 32 * cc, r);
        }
      }
      // P (fp16) over S; hi+lo split for rows that see few keys
      {
        uint32_t r[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = pack_f16x2(s[64 * cc + 2 * i], s[64 * cc + 2 * i + 1]);
          tmem_st32(tS + 32 * cc, r);
        }
        if (hilo) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a0 = s[64 * cc + 2 * i], a1 = s[64 * cc + 2 * i + 1];
              const uint32_t hi2 = pack_f16x2(a0, a1);
              r[i] = pack_f16x2(a0 - f16_lo_to_f32(hi2), a1 - f16_hi_to_f32(hi2));
            }
            tmem_st32(tS + 64 + 32 * cc, r);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR_PFULL(t));
    }
    // ---------------------------------------------------------- epilogue
    if (qt < p.n_qt && ok) {
      bool acc = false;
      if (nt > 0) {
        acc = __all_sync(0xffffffffu, wait_bar(BAR_OREADY(t), (nt - 1) & 1, wc));
        tc_fence_after();
      }
      const bool write = qi < p.Sq && (nt == 0 || acc);
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((size_t)(b * p.Hq + h) * p.Sq + qi) * Dv;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < Dv / 32; ++cc) {
        uint32_t r[32];
        if (acc) {
          tmem_ld32(tO + 32 * cc, r);   // warp-collective: all lanes, even rows past Sq
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = __uint_as_float(r[2 * i]) * inv_l;
          const float a1 = __uint_as_float(r[2 * i + 1]) * inv_l;
          w[i] = kBF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
        }
        if (write) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (write)
        p.lse[(size_t)(b * p.Hq + h) * p.Sq + qi] = (l > 0.f) ? m * p.scale + __logf(l) : INFINITY;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
