// Elementwise kernels of the backward that materialises S, P, dP and dS per
// (KV head, head of its group), with every product a tensor-core GEMM of the
// inputs' 16-bit type accumulated in fp32; P and dS enter the products as
// hi + lo pairs of that type:
//   S = Q K^T,  P = exp(scale S - LSE),  dV += P^T dO,  dP = dO V^T,
//   dS = P * (dP - d_row),  dQ = scale dS K,  dK += scale dS^T Q
// (the steps of the BSA PyPTO implementation notes' backward: section 3.2
// "Core design strategies", P recomputed from the forward's LSE; section 8.4,
// d_row = rowsum(dO * O) computed once beforehand; section 1, dV unscaled,
// dQ and dK scaled).  A batch of the GEMMs covers `planes` KV planes p (batch
// b = p / Hkv) at one head g of each group, i.e. query planes p * G + g.
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

// 16-bit operands of the tensor-core products: P = exp(scale * s - LSE), 0 on
// masked keys, rows past the batch's length and rows without keys, split into
// hi = P rounded to the inputs' type and lo = (P - hi) rounded, written to two
// matrices of the batch's layout.  kV elements per thread and step: 8 (32-byte
// loads, 16-byte stores) when Skv and ncols are multiples of 8, else 1.
// Grid: (rows of the block, planes).
template <bool kBF16>
__device__ __forceinline__ float h16_to_f32(uint32_t h) {
  return kBF16 ? __uint_as_float(h << 16) : f16_lo_to_f32(h);
}
template <bool kBF16>
__device__ __forceinline__ void split_hilo(float x, uint32_t& hi, uint32_t& lo) {
  hi = (kBF16 ? pack_bf16x2(x, 0.f) : pack_f16x2(x, 0.f)) & 0xFFFFu;
  const float r = x - h16_to_f32<kBF16>(hi);
  lo = (kBF16 ? pack_bf16x2(r, 0.f) : pack_f16x2(r, 0.f)) & 0xFFFFu;
}
template <bool kBF16, int kV>
__global__ void __launch_bounds__(256) fa_bwd_p_hilo_kernel(const float* __restrict__ s,
                                                            uint16_t* __restrict__ ph,
                                                            uint16_t* __restrict__ pl,
                                                            BwdGemmRows r) {
  const int i = r.row0 + blockIdx.x;
  const int z = blockIdx.y;
  const int p = r.plane0 + z;
  const int b = p / r.Hkv;
  const int q_len = r.seqlens ? min(r.seqlens[b], r.Sq) : r.Sq;
  const int kv_len = r.seqlens ? min(r.seqlens[b], r.Skv) : r.Skv;
  const float lse = r.lse[(size_t)(p * r.G + r.g) * r.Sq + i];
  const bool row_ok = i < q_len && lse != INFINITY;
  int lim = row_ok ? kv_len : 0;
  if (r.causal) lim = min(lim, i + 1);
  const size_t base = ((size_t)z * r.Sq + i) * r.Skv;
  for (int j0 = threadIdx.x * kV; j0 < r.ncols; j0 += blockDim.x * kV) {
    float x[kV];
    if constexpr (kV == 8) {
      const float4 a = *reinterpret_cast<const float4*>(s + base + j0);
      const float4 c = *reinterpret_cast<const float4*>(s + base + j0 + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
    } else {
      x[0] = s[base + j0];
    }
    uint32_t h[kV], l[kV];
#pragma unroll
    for (int e = 0; e < kV; ++e)
      split_hilo<kBF16>(j0 + e < lim ? expf(fmaf(x[e], r.scale, -lse)) : 0.f, h[e], l[e]);
    if constexpr (kV == 8) {
      *reinterpret_cast<uint4*>(ph + base + j0) =
          make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
      *reinterpret_cast<uint4*>(pl + base + j0) =
          make_uint4(l[0] | l[1] << 16, l[2] | l[3] << 16, l[4] | l[5] << 16, l[6] | l[7] << 16);
    } else {
      ph[base + j0] = (uint16_t)h[0];
      pl[base + j0] = (uint16_t)l[0];
    }
  }
}

// dS = P * (dP - d_row) with P = hi + lo read from the pair, written back over
// the pair as hi and lo of the inputs' type; exactly 0 where P is (masked
// keys, padded rows: whatever dO holds there cannot reach dQ, dK or dV).  An
// fp16 dS beyond the fp16 range sets kStatusRange.  kV as above.
// Grid: (rows of the block, planes).
template <bool kBF16, int kV>
__global__ void __launch_bounds__(256) fa_bwd_ds_hilo_kernel(uint16_t* __restrict__ ph,
                                                             uint16_t* __restrict__ pl,
                                                             const float* __restrict__ dp,
                                                             BwdGemmRows r) {
  const int i = r.row0 + blockIdx.x;
  const int z = blockIdx.y;
  const int p = r.plane0 + z;
  const float d = r.d_row[(size_t)(p * r.G + r.g) * r.Sq + i];
  const size_t base = ((size_t)z * r.Sq + i) * r.Skv;
  for (int j0 = threadIdx.x * kV; j0 < r.ncols; j0 += blockDim.x * kV) {
    float pv[kV], dv[kV];
    if constexpr (kV == 8) {
      const uint4 hh = *reinterpret_cast<const uint4*>(ph + base + j0);
      const uint4 ll = *reinterpret_cast<const uint4*>(pl + base + j0);
      const uint32_t hw[4] = {hh.x, hh.y, hh.z, hh.w}, lw[4] = {ll.x, ll.y, ll.z, ll.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[2 * e] = h16_to_f32<kBF16>(hw[e] & 0xFFFFu) + h16_to_f32<kBF16>(lw[e] & 0xFFFFu);
        pv[2 * e + 1] = h16_to_f32<kBF16>(hw[e] >> 16) + h16_to_f32<kBF16>(lw[e] >> 16);
      }
      const float4 a = *reinterpret_cast<const float4*>(dp + base + j0);
      const float4 c = *reinterpret_cast<const float4*>(dp + base + j0 + 4);
      dv[0] = a.x; dv[1] = a.y; dv[2] = a.z; dv[3] = a.w;
      dv[4] = c.x; dv[5] = c.y; dv[6] = c.z; dv[7] = c.w;
    } else {
      pv[0] = h16_to_f32<kBF16>(ph[base + j0]) + h16_to_f32<kBF16>(pl[base + j0]);
      dv[0] = dp[base + j0];
    }
    uint32_t h[kV], l[kV];
    bool big = false;
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const float x = pv[e] != 0.f ? pv[e] * (dv[e] - d) : 0.f;
      if (!kBF16) big |= !(fabsf(x) <= 65504.f);
      split_hilo<kBF16>(x, h[e], l[e]);
    }
    if (!kBF16 && big) atomicOr(r.status, kStatusRange);
    if constexpr (kV == 8) {
      *reinterpret_cast<uint4*>(ph + base + j0) =
          make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
      *reinterpret_cast<uint4*>(pl + base + j0) =
          make_uint4(l[0] | l[1] << 16, l[2] | l[3] << 16, l[4] | l[5] << 16, l[6] | l[7] << 16);
    } else {
      ph[base + j0] = (uint16_t)h[0];
      pl[base + j0] = (uint16_t)l[0];
    }
  }
}

}  // namespace fa
