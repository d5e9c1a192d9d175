// Elementwise kernels of the backward that materialises S, P, dP and dS per
// (KV head, head of its group), with every product a tensor-core GEMM of the
// inputs' 16-bit type accumulated in fp32:
//   S = Q K^T,  dP = dO V^T,  P = exp(scale S - LSE),  dS = P * (dP - d_row),
//   dV += P^T dO,  dQ = scale dS K,  dK += scale dS^T Q
// (the steps of the BSA PyPTO implementation notes' backward: section 3.2
// "Core design strategies", P recomputed from the forward's LSE; section 8.4,
// d_row = rowsum(dO * O) computed once beforehand; section 1, dV unscaled,
// dQ and dK scaled).  A batch of the GEMMs covers `planes` KV planes p (batch
// b = p / Hkv) at one head g of each group, i.e. query planes p * G + g.
//
// P and dS enter their products as hi + lo pairs of the inputs' type (hi =
// round(x), lo = round(x - hi)), written in place over the fp32 S and dP:
// element j of a row becomes the 16-bit values 2j (hi) and 2j + 1 (lo).  Read
// as 16-bit, a row of the fp32 buffer is a row of 2 ncols interleaved values
// (leading dimension 2 Skv), so each product takes the pair in one GEMM with
// a doubled inner or outer dimension:
//   dV2 += P2^T dO,  dK2 += scale dS2^T Q   (2 Skv rows: row 2j + e holds
//                                            the hi (e = 0) or lo part of key j)
//   dQ = scale dS2 K2                        (K2: every row of K twice)
// and dV, dK are the sums of the row pairs of dV2, dK2.
#pragma once
#include "fa_ptx.cuh"

namespace fa {

// fp32 -> bf16 or fp16 (round to nearest even), n8 groups of 8 elements.
template <bool kBF16>
__global__ void __launch_bounds__(256) fa_bwd_from_f32_kernel(const float4* __restrict__ in,
                                                              uint4* __restrict__ out, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = in[2 * i], c = in[2 * i + 1];
    out[i] = kBF16 ? make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(c.x, c.y),
                                pack_bf16x2(c.z, c.w))
                   : make_uint4(pack_f16x2(a.x, a.y), pack_f16x2(a.z, a.w), pack_f16x2(c.x, c.y),
                                pack_f16x2(c.z, c.w));
  }
}

// out[r, :] = round(in[2r, :] + in[2r + 1, :]) for rows of D fp32 values
// (D a multiple of 8), n8 groups of 8 output elements.
template <bool kBF16>
__global__ void __launch_bounds__(256) fa_bwd_from_f32_pairs_kernel(const float4* __restrict__ in,
                                                                    uint4* __restrict__ out,
                                                                    size_t n8, int D) {
  const size_t g_row = (size_t)D / 8;   // groups of 8 per row
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / g_row, c8 = i - r * g_row;
    const float4* a = in + (2 * r * g_row + c8) * 2;    // row 2r, group c8
    const float4* b = a + g_row * 2;                    // row 2r + 1
    const float4 a0 = a[0], a1 = a[1], b0 = b[0], b1 = b[1];
    const float x0 = a0.x + b0.x, x1 = a0.y + b0.y, x2 = a0.z + b0.z, x3 = a0.w + b0.w;
    const float x4 = a1.x + b1.x, x5 = a1.y + b1.y, x6 = a1.z + b1.z, x7 = a1.w + b1.w;
    out[i] = kBF16 ? make_uint4(pack_bf16x2(x0, x1), pack_bf16x2(x2, x3), pack_bf16x2(x4, x5),
                                pack_bf16x2(x6, x7))
                   : make_uint4(pack_f16x2(x0, x1), pack_f16x2(x2, x3), pack_f16x2(x4, x5),
                                pack_f16x2(x6, x7));
  }
}

// K2: every row of D 16-bit values written twice (rows 2r and 2r + 1), n8
// groups of 8 input elements (D a multiple of 8).
__global__ void __launch_bounds__(256) fa_bwd_dup_rows_kernel(const uint4* __restrict__ in,
                                                              uint4* __restrict__ out, size_t n8,
                                                              int D) {
  const size_t g_row = (size_t)D / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / g_row, c8 = i - r * g_row;
    const uint4 v = in[i];
    out[2 * r * g_row + c8] = v;
    out[(2 * r + 1) * g_row + c8] = v;
  }
}

struct BwdGemmRows {
  const float* lse;      // [B * Hq * Sq], natural-log units (+inf on rows without keys)
  const float* d_row;    // [B * Hq * Sq]
  const int* seqlens;    // per-batch lengths, or null
  int Hkv, G, Sq, Skv;
  int causal;            // top-left: key j is seen by row i iff j <= i
  float scale;
  int plane0;            // first KV plane of the batch of GEMMs
  int g;                 // head of the group
  int row0;              // first row of the row block (grid.x counts rows from here)
  int ncols;             // keys [0, ncols) of the block's rows are written (the rest unused)
  int* status;           // fp16 pairs: kStatusRange when a dS value is beyond the fp16 range
};

template <bool kBF16>
__device__ __forceinline__ uint32_t split_hilo(float x) {   // hi | lo << 16
  const uint32_t hi = (kBF16 ? pack_bf16x2(x, 0.f) : pack_f16x2(x, 0.f)) & 0xFFFFu;
  const float h = kBF16 ? __uint_as_float(hi << 16) : f16_lo_to_f32(hi);
  const uint32_t lo = (kBF16 ? pack_bf16x2(x - h, 0.f) : pack_f16x2(x - h, 0.f)) & 0xFFFFu;
  return hi | lo << 16;
}

// P = exp(scale * s - LSE), 0 on masked keys, rows past the batch's length
// and rows without keys; dS = P * (dP - d_row), exactly 0 where P is (masked
// keys, padded rows: whatever dO holds there cannot reach dQ, dK or dV).  Both
// written in place as pairs over the fp32 S and dP.  An fp16 dS beyond the
// fp16 range sets kStatusRange.  kV elements per thread and step: 8 (32-byte
// loads and stores) when Skv and ncols are multiples of 8, else 1.
// Grid: (rows of the block, planes).
template <bool kBF16, int kV>
__global__ void __launch_bounds__(256) fa_bwd_p_ds_kernel(float* __restrict__ s,
                                                          float* __restrict__ dp,
                                                          BwdGemmRows r) {
  const int i = r.row0 + blockIdx.x;
  const int z = blockIdx.y;
  const int p = r.plane0 + z;
  const int b = p / r.Hkv;
  const int q_len = r.seqlens ? min(r.seqlens[b], r.Sq) : r.Sq;
  const int kv_len = r.seqlens ? min(r.seqlens[b], r.Skv) : r.Skv;
  const size_t row = (size_t)(p * r.G + r.g) * r.Sq + i;
  const float lse = r.lse[row];
  const float d = r.d_row[row];
  const bool row_ok = i < q_len && lse != INFINITY;
  int lim = row_ok ? kv_len : 0;
  if (r.causal) lim = min(lim, i + 1);
  const size_t base = ((size_t)z * r.Sq + i) * r.Skv;
  bool big = false;
  for (int j0 = threadIdx.x * kV; j0 < r.ncols; j0 += blockDim.x * kV) {
    float x[kV], y[kV];
    if (j0 >= lim) {   // every key of the group masked: zero pairs, S and dP not read
      if constexpr (kV == 8) {
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(s + base + j0) = zero;
        *reinterpret_cast<uint4*>(s + base + j0 + 4) = zero;
        *reinterpret_cast<uint4*>(dp + base + j0) = zero;
        *reinterpret_cast<uint4*>(dp + base + j0 + 4) = zero;
      } else {
        reinterpret_cast<uint32_t*>(s)[base + j0] = 0u;
        reinterpret_cast<uint32_t*>(dp)[base + j0] = 0u;
      }
      continue;
    }
    if constexpr (kV == 8) {
      const float4 a = *reinterpret_cast<const float4*>(s + base + j0);
      const float4 c = *reinterpret_cast<const float4*>(s + base + j0 + 4);
      const float4 e = *reinterpret_cast<const float4*>(dp + base + j0);
      const float4 f = *reinterpret_cast<const float4*>(dp + base + j0 + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
      y[0] = e.x; y[1] = e.y; y[2] = e.z; y[3] = e.w; y[4] = f.x; y[5] = f.y; y[6] = f.z; y[7] = f.w;
    } else {
      x[0] = s[base + j0];
      y[0] = dp[base + j0];
    }
    uint32_t pw[kV], dw[kV];
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const float pv = j0 + e < lim ? expf(fmaf(x[e], r.scale, -lse)) : 0.f;
      const float ds = pv != 0.f ? pv * (y[e] - d) : 0.f;
      if (!kBF16) big |= !(fabsf(ds) <= 65504.f);
      pw[e] = split_hilo<kBF16>(pv);
      dw[e] = split_hilo<kBF16>(ds);
    }
    if constexpr (kV == 8) {
      *reinterpret_cast<uint4*>(s + base + j0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(s + base + j0 + 4) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      *reinterpret_cast<uint4*>(dp + base + j0) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      *reinterpret_cast<uint4*>(dp + base + j0 + 4) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
    } else {
      reinterpret_cast<uint32_t*>(s)[base + j0] = pw[0];
      reinterpret_cast<uint32_t*>(dp)[base + j0] = dw[0];
    }
  }
  if (!kBF16 && big) atomicOr(r.status, kStatusRange);
}

}  // namespace fa
