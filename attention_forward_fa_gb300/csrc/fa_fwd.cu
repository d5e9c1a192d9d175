// Host side of libfa_fwd.so: argument validation, TMA descriptors, variant
// selection and launch.  The C ABI is declared in include/fa_fwd.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>
#include <algorithm>
#include <mutex>

#include "../../include/fa_fwd.h"
#include "fa_tiled.cuh"
#include "fa_mla.cuh"
#include "fa_bwd.cuh"
#include "fa_bwd_gemm.cuh"

#include <cublas_v2.h>

namespace {

// Device status word of this module (one per device the library runs on):
// bit 0 = a bounded wait expired, bit 1 = a bf16 V value overflowed fp16.
__device__ int g_fa_status;

// Fixed scratch of fa_fwd_noalloc, kNoAllocScratchBytes long.  It holds either
// the fp16 copy of a bf16 key latent (top-k calls) or the fp32 O / l and LSE
// pieces of a dense call split along its KV tiles; any two fa_fwd_noalloc calls
// that overlap on the GPU therefore race on it, whatever their kinds.  It is
// part of the module image, so every device that loads this library holds it
// until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<int> g_last_cuda{0};
#ifdef FA_TRACE
unsigned long long* g_trace = nullptr;
#endif
std::atomic<long long> g_timeout_ns{2000000000LL};
std::atomic<int> g_max_kv_split{fa::kMaxSplit};   // pieces per unit at most (1: never split)

// Device address of g_noalloc_scratch for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
static void* noalloc_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) {
      g_last_cuda.store((int)e);
      return nullptr;
    }
    addr[dev] = ptr;
  }
  return addr[dev];
}

int cuda_fail(cudaError_t e) {
  g_last_cuda.store((int)e);
  return FA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D view (cols, rows, planes) of a contiguous [planes, rows, cols] 16-bit
// tensor, tiled in boxes of 64 columns x box_rows rows x box_planes planes with
// 128-byte swizzle.
bool encode_3d(CUtensorMap* tm, const void* base, bool fp16, uint64_t cols, uint64_t rows,
               uint64_t planes, uint32_t box_rows, uint32_t box_planes = 1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, box_rows, box_planes};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int* status_ptr() {
  // the symbol's device address for the current device
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_fa_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(ptr);
}

// bf16 -> fp16 copy of V (the P.V product runs on fp16 operands; fp16 keeps
// three more mantissa bits of P than bf16).  bf16 -> fp16 is exact for
// 2^-14 <= |v| <= 65504; larger magnitudes become inf and set status bit 1.
__global__ void __launch_bounds__(256) fa_convert_v_kernel(const uint4* __restrict__ in,
                                                            uint4* __restrict__ out, size_t n16,
                                                            int* status) {
  constexpr int kUnroll = 4;   // 16-byte loads in flight per thread
  uint32_t vmax = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = __ldcs(in + i + u * stride);   // read once
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      uint32_t* ww = reinterpret_cast<uint32_t*>(&w[u]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        vmax = fa::max_u16x2(vmax, ww[q] & 0x7FFF7FFFu);
        ww[q] = fa::pack_f16x2(__uint_as_float(ww[q] << 16), __uint_as_float(ww[q] & 0xFFFF0000u));
      }
      out[i + u * stride] = w[u];
    }
  }
  for (; i < n16; i += stride) {
    uint4 w = in[i];
    uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      vmax = fa::max_u16x2(vmax, ww[q] & 0x7FFF7FFFu);
      ww[q] = fa::pack_f16x2(__uint_as_float(ww[q] << 16), __uint_as_float(ww[q] & 0xFFFF0000u));
    }
    out[i] = w;
  }
  if ((vmax & 0xFFFFu) > 0x477Fu || (vmax >> 16) > 0x477Fu) atomicOr(status, fa::kStatusRange);
}

// FP8 inputs as fp16: the values of x_q (e4m3fn or e5m2 bytes), exact since
// both formats lie inside fp16 (d_scale null; the attention kernel applies the
// dequant scales), or x_q * d_scale of the row's block of 128 rows along S
// rounded once to fp16.  x_q [planes, S, D], d_scale [planes, ceil(S / 128)].
// Each thread converts 16 bytes.
template <bool E5M2>
__global__ void __launch_bounds__(256) fa_fp8_to_fp16_kernel(const uint4* __restrict__ in,
                                                             const float* __restrict__ d_scale,
                                                             uint4* __restrict__ out, size_t n16,
                                                             int S, int D) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const int nb = (S + 127) / 128;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
    float d = 1.f;
    if (d_scale) {
      const size_t row = (i * 16) / (size_t)D;            // D is a multiple of 16
      const size_t plane = row / (size_t)S;
      d = d_scale[plane * nb + (int)(row - plane * S) / 128];
    }
    const uint4 w = in[i];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint16_t two = (uint16_t)(ww[q] >> (16 * e));
        uint32_t f2;
        if (E5M2)
          asm("{\n .reg .b16 t;\n mov.b16 t, %1;\n cvt.rn.f16x2.e5m2x2 %0, t;\n}" : "=r"(f2) : "h"(two));
        else
          asm("{\n .reg .b16 t;\n mov.b16 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(f2) : "h"(two));
        h[2 * q + e] = d_scale ? fa::pack_f16x2(fa::f16_lo_to_f32(f2) * d, fa::f16_hi_to_f32(f2) * d) : f2;
      }
    }
    out[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

int fp8_to_fp16(const void* x8, const float* d_scale, void* x16, size_t planes, int S, int D,
                bool e5m2, cudaStream_t st) {
  const size_t n16 = planes * (size_t)S * D / 16;   // D is a multiple of 16
  int blocks = (int)std::min<size_t>((n16 + 255) / 256, 152 * 8);
  if (blocks < 1) blocks = 1;
  if (e5m2)
    fa_fp8_to_fp16_kernel<true><<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x8), d_scale,
                                                        static_cast<uint4*>(x16), n16, S, D);
  else
    fa_fp8_to_fp16_kernel<false><<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x8), d_scale,
                                                         static_cast<uint4*>(x16), n16, S, D);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int convert_v(const void* v, void* vh, size_t n_elems, int* status, cudaStream_t st) {
  const size_t n16 = n_elems / 8;
  int blocks = (int)std::min<size_t>((n16 + 255) / 256, 152 * 8);
  if (blocks < 1) blocks = 1;
  fa_convert_v_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(v), static_cast<uint4*>(vh),
                                              n16, status);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

// Stream-ordered scratch from the device's default memory pool, which is
// told once to keep freed blocks cached (no release at synchronisation).
void* scratch_alloc(size_t bytes, cudaStream_t st) {
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [dev] {
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      uint64_t thr = ~0ull;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
  });
  void* ptr = nullptr;
  if (cudaMallocAsync(&ptr, bytes, st) != cudaSuccess) return nullptr;
  return ptr;
}

// Merge of the pieces of split units, the blockwise merge of the pages in LSE
// form: one warp per output row, O = sum_p exp(LSE_p - LSE) O_p with
// LSE = m + ln sum_p exp(LSE_p - m), m = max_p LSE_p; a row that no piece saw
// a key of gets O = 0 and LSE = +inf.  Launched as a programmatic dependent of
// the tiled kernel: it may be scheduled while that kernel drains and waits for
// it before reading the pieces.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_merge_kernel(const float* __restrict__ part_o,
                                                       const float* __restrict__ part_lse,
                                                       void* __restrict__ o,
                                                       void* __restrict__ o_lo,
                                                       float* __restrict__ lse, long long rows,
                                                       int Dv, int nsplit) {
  fa::pdl_launch_dependents();
  fa::pdl_wait_prior();
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float lp[fa::kMaxSplit];
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < fa::kMaxSplit; ++s) {
    lp[s] = s < nsplit ? part_lse[(size_t)s * rows + row] : -INFINITY;
    m = fmaxf(m, lp[s]);
  }
  const bool empty = !(m > -INFINITY);
  float w[fa::kMaxSplit];
  float L = 0.f;
#pragma unroll
  for (int s = 0; s < fa::kMaxSplit; ++s) {
    w[s] = empty ? 0.f : expf(lp[s] - m);   // 0 for a piece without keys
    L += w[s];
  }
  const float inv = empty ? 0.f : 1.f / L;
  for (int c = 4 * lane; c < Dv; c += 128) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < fa::kMaxSplit; ++s) {
      if (w[s] == 0.f) continue;
      const float4 x = *reinterpret_cast<const float4*>(part_o + ((size_t)s * rows + row) * Dv + c);
      a.x = fmaf(w[s], x.x, a.x);
      a.y = fmaf(w[s], x.y, a.y);
      a.z = fmaf(w[s], x.z, a.z);
      a.w = fmaf(w[s], x.w, a.w);
    }
    const float x0 = a.x * inv, x1 = a.y * inv, x2 = a.z * inv, x3 = a.w * inv;
    uint2 pk;
    pk.x = BF16 ? fa::pack_bf16x2(x0, x1) : fa::pack_f16x2(x0, x1);
    pk.y = BF16 ? fa::pack_bf16x2(x2, x3) : fa::pack_f16x2(x2, x3);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(o) + ((size_t)row * Dv + c) * 2) = pk;
    if (o_lo)
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(o_lo) + ((size_t)row * Dv + c) * 2) =
          make_uint2(fa::pack_residual_x2(x0, x1, pk.x, BF16), fa::pack_residual_x2(x2, x3, pk.y, BF16));
  }
  if (lane == 0) lse[row] = empty ? INFINITY : m + logf(L);
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
  static int sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) sms[dev] = n;
  }
  return sms[dev];
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel on the stream drains; it waits for that kernel
// (griddepcontrol.wait) before its first global memory access.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, bool BF16, int NS, bool CONV, bool SPLIT, bool EXTRAS = false>
int launch_tiled(const fa::TiledParams& prm, int units, cudaStream_t st) {
  auto kern = fa::fa_fwd_tiled_kernel<D, BF16, NS, CONV, SPLIT, EXTRAS>;
  constexpr int smem = fa::TiledSmem<D, NS>::kAlloc;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  static int regs_ok[64];
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    // The warpgroups re-split the register file with setmaxnreg; that only
    // works if every thread was launched with at least the average of the
    // split (an unmet setmaxnreg.inc would wait forever).
    cudaFuncAttributes fattr;
    if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fattr, kern);
    if (attr_err == cudaSuccess) regs_ok[dev & 63] = fattr.numRegs >= fa::kRegsNeeded ? 1 : -1;
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err);
  if (regs_ok[dev & 63] != 1) return cuda_fail(cudaErrorInvalidConfiguration);
  cudaError_t e = launch_dependent(kern, (unsigned)units, fa::kTiledThreads, smem, st, prm);
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// The dense kernel for (head dim, input type, V conversion), split or not,
// with the optional terms or not.
template <bool SPLIT, bool EXTRAS = false>
int launch_tiled_variant(const fa::TiledParams& prm, int grid, cudaStream_t st, int D, bool fp16,
                         bool conv) {
  if (D == 128) {
    if (fp16) return launch_tiled<128, false, 4, false, SPLIT, EXTRAS>(prm, grid, st);
    return conv ? launch_tiled<128, true, 4, true, SPLIT, EXTRAS>(prm, grid, st)
                : launch_tiled<128, true, 4, false, SPLIT, EXTRAS>(prm, grid, st);
  }
  if (fp16) return launch_tiled<64, false, 6, false, SPLIT, EXTRAS>(prm, grid, st);
  return conv ? launch_tiled<64, true, 6, true, SPLIT, EXTRAS>(prm, grid, st)
              : launch_tiled<64, true, 6, false, SPLIT, EXTRAS>(prm, grid, st);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Argument checks shared by the entry points (nothing is launched on error).
int validate(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
             const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
             const fa_topk_t* topk_idx, float rescale_threshold) {
  const int mask = mask_mode & 0xF;
  const bool v_from_k = (mask_mode & FA_V_FROM_K) != 0;
  if (mask_mode & ~(0xF | FA_DTYPE_FP16 | FA_V_FROM_K | FA_V_FP16)) return FA_ERR_SHAPE;
  // ---- pointers
  if (!q || !k || !o || !lse || (!v && !v_from_k)) return FA_ERR_NULL;
  if (kv_block_idx && !kv_block_idx->idx) return FA_ERR_NULL;
  if (topk_idx && !topk_idx->idx) return FA_ERR_NULL;
  // ---- shapes
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0 || Dv <= 0)
    return FA_ERR_SHAPE;
  if (Hq % Hkv) return FA_ERR_SHAPE;
  if (kv_block_idx && topk_idx) return FA_ERR_SHAPE;
  if (mask > FA_MASK_CAUSAL_DIAG_BLOCK) return FA_ERR_SHAPE;
  if (mask == FA_MASK_CAUSAL_DIAG_BLOCK && !kv_block_idx) return FA_ERR_SHAPE;
  if (kv_block_idx) {
    if (kv_block_idx->block != 128) return FA_ERR_SHAPE;
    if (kv_block_idx->max_sel <= 0 || kv_block_idx->max_sel > fa::kMaxSel) return FA_ERR_SHAPE;
    if (kv_block_idx->stride_b < 0 || kv_block_idx->stride_h < 0) return FA_ERR_SHAPE;
  }
  if (topk_idx && (topk_idx->topk <= 0 || topk_idx->topk > fa::kMlaMaxTopk ||
                   topk_idx->stride_b < 0))
    return FA_ERR_SHAPE;
  if (!std::isfinite(scale)) return FA_ERR_SHAPE;
  if (!(rescale_threshold >= 0.f && rescale_threshold <= 15.f)) return FA_ERR_THRESHOLD;
  if ((long long)B * Hq > (1LL << 30) || (long long)Sq * 128 > (1LL << 31) ||
      (long long)Skv * 128 > (1LL << 31))
    return FA_ERR_SHAPE;
  // ---- supported variants
  const bool tiled = !topk_idx && !v_from_k && D == Dv && (D == 64 || D == 128);
  const bool mla = topk_idx && v_from_k && D == fa::kMlaD && Dv == fa::kMlaDv && Hkv == 1;
  if (!tiled && !mla) return FA_ERR_UNSUPPORTED;
  if (mla) {
    const long long units = (long long)B * Sq * ((Hq + fa::kMlaHeads - 1) / fa::kMlaHeads);
    if ((long long)B * Skv > 0x7FFFFFFFLL || units * fa::kMlaSplit > 0x7FFFFFFFLL)
      return FA_ERR_SHAPE;
  }
  // ---- alignment (TMA: 16-byte bases; vector stores of O)
  if (!aligned(q, 16) || !aligned(k, 16) || (v && !aligned(v, 16)) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_ALIGN;
  if (seqlens && !aligned(seqlens, 4)) return FA_ERR_ALIGN;
  if (kv_block_idx && !aligned(kv_block_idx->idx, 4)) return FA_ERR_ALIGN;
  if (topk_idx && !aligned(topk_idx->idx, 4)) return FA_ERR_ALIGN;
  return FA_OK;
}

// Checks of the optional terms (fa_fwd_ext, fa_fwd_fp8); nothing is launched.
int validate_extras(const fa_extras_t* extras, int Skv) {
  if (extras->window < 0 || extras->window > 2 || extras->alibi < 0 || extras->alibi > 2)
    return FA_ERR_SHAPE;
  if ((Skv + fa::kBN - 1) / fa::kBN > fa::kMaxSel) return FA_ERR_SHAPE;
  // keep_prob 0 (a zero-initialised struct) or 1: no dropout
  if (!(extras->keep_prob >= 0.f && extras->keep_prob <= 1.f)) return FA_ERR_SHAPE;
  const bool dropout = extras->keep_prob > 0.f && extras->keep_prob < 1.f;
  if (dropout && (extras->offset % 16 || Skv % 16)) return FA_ERR_SHAPE;
  if (extras->pse) {
    if (extras->alibi || extras->pse_type < 0 || extras->pse_type > 1) return FA_ERR_SHAPE;
    if (extras->pse_stride_b < 0 || extras->pse_stride_h < 0 || extras->pse_stride_q < 0)
      return FA_ERR_SHAPE;
    if (!aligned(extras->pse, 16) || extras->pse_stride_q % 8 || extras->pse_stride_h % 8 ||
        extras->pse_stride_b % 8 || Skv % 8)
      return FA_ERR_ALIGN;
  }
  if (extras->atten_mask) {
    if (extras->mask_stride_b < 0 || extras->mask_stride_h < 0 || extras->mask_stride_q < 0)
      return FA_ERR_SHAPE;
    if (!aligned(extras->atten_mask, 16) || extras->mask_stride_q % 16 ||
        extras->mask_stride_h % 16 || extras->mask_stride_b % 16 || Skv % 16)
      return FA_ERR_ALIGN;
  }
  return FA_OK;
}

template <bool BF16>
int launch_mla(const fa::MlaParams& prm, long long units, cudaStream_t st) {
  auto kern = fa::fa_mla_topk_kernel<BF16>;
  constexpr int smem = fa::MlaSmem::kAlloc;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_err[64];
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err[dev & 63] != cudaSuccess) return cuda_fail(attr_err[dev & 63]);
  cudaError_t e = launch_dependent(kern, (unsigned)units, fa::kMlaThreads, smem, st, prm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

// Top-k sparse MLA forward on validated arguments; `k16` is the key latent
// [B, Skv, 576] in fp16 (the caller's for fp16 inputs or with FA_V_FP16, a
// converted copy otherwise).
int run_topk(const void* q, const void* k16, void* o, void* o_lo, float* lse, int B, int Hq,
             int Sq, int Skv, float scale, int mask_mode, const int32_t* seqlens,
             const fa_topk_t* tk, float rescale_threshold, int* status, cudaStream_t st) {
  const bool fp16 = (mask_mode & FA_DTYPE_FP16) != 0;
  fa::MlaParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const uint32_t q_rows = (uint32_t)std::min<long long>(fa::kMlaHeads, (long long)B * Hq);
  if (!encode_3d(&prm.tm_q, q, fp16, fa::kMlaD, Sq, (uint64_t)B * Hq, 1, q_rows))
    return cuda_fail(cudaErrorInvalidValue);
  prm.kl = static_cast<const uint16_t*>(k16);
  prm.q_rows = (int)q_rows;
  prm.o = o;
  prm.o_lo = o_lo;
  prm.lse = lse;
  prm.seqlens = seqlens;
  prm.topk = tk->idx;
  prm.topk_stride_b = tk->stride_b;
  prm.W = tk->topk;
  prm.B = B;
  prm.Hq = Hq;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.n_hg = (Hq + fa::kMlaHeads - 1) / fa::kMlaHeads;
  prm.causal = (mask_mode & 0xF) == FA_MASK_CAUSAL;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.threshold = rescale_threshold;
  prm.timeout_ns = g_timeout_ns.load();
  prm.status = status;
  const long long units = (long long)B * Sq * prm.n_hg * fa::kMlaSplit;
  return fp16 ? launch_mla<false>(prm, units, st) : launch_mla<true>(prm, units, st);
}

// Tiled forward on validated arguments.  `v` is fp16 (fp16 inputs, or a bf16
// call with FA_V_FP16), else bf16, converted tile by tile inside the kernel.
int run_tiled(const void* q, const void* k, const void* v, void* o, void* o_lo, float* lse, int B,
              int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
              const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
              float rescale_threshold, int* status, cudaStream_t st, bool may_alloc,
              const fa_extras_t* ex = nullptr, const float* ds_q = nullptr,
              const float* ds_k = nullptr, const float* ds_v = nullptr) {
  const int mask = mask_mode & 0xF;
  const bool fp16 = (mask_mode & FA_DTYPE_FP16) != 0;
  const bool conv = !fp16 && !(mask_mode & FA_V_FP16);   // V arrives as bf16
  fa::TiledParams prm;
  std::memset(&prm, 0, sizeof(prm));
  if (!encode_3d(&prm.tm_q, q, fp16, D, Sq, (uint64_t)B * Hq, fa::kBM) ||
      !encode_3d(&prm.tm_k, k, fp16, D, Skv, (uint64_t)B * Hkv, fa::kBN) ||
      !encode_3d(&prm.tm_v, v, /*fp16=*/!conv, Dv, Skv, (uint64_t)B * Hkv, fa::kBN))
    return cuda_fail(cudaErrorInvalidValue);
  prm.o = o;
  prm.o_lo = o_lo;
  prm.lse = lse;
  prm.seqlens = seqlens;
  if (kv_block_idx) {
    prm.blk_idx = kv_block_idx->idx;
    prm.blk_stride_b = kv_block_idx->stride_b;
    prm.blk_stride_h = kv_block_idx->stride_h;
    prm.max_sel = kv_block_idx->max_sel;
  }
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.mask = mask;
  prm.n_qt = (Sq + fa::kBM - 1) / fa::kBM;
  // Slot pairing: two heads of one GQA group at the same query tile when the
  // group size is even (identical KV sequence), else two consecutive query
  // tiles of one head.  Block lists that differ per head or per query block
  // simply give the two slots independent KV sequences.
  const bool head_pairs = (prm.G % 2 == 0);
  prm.pair_mode = head_pairs ? 1 : 0;
  if (head_pairs) {
    prm.units_per_q = B * (Hq / 2);
    prm.n_qpos = prm.n_qt;
  } else {
    prm.units_per_q = B * Hq;
    prm.n_qpos = (prm.n_qt + 1) / 2;
  }
  // block lists: one head's units after another (unit_of in fa_tiled.cuh)
  prm.head_major = kv_block_idx ? 1 : 0;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.threshold = rescale_threshold;
  prm.timeout_ns = g_timeout_ns.load();
  prm.status = status;
#ifdef FA_TRACE
  prm.trace = g_trace;
#endif
  if (ex) {
    // window bounds beyond +-(Sq + Skv) cannot change a row's key range
    const long long lim = (long long)Sq + Skv;
    auto clampw = [lim](int32_t v) { return (int)std::max(-lim, std::min(lim, (long long)v)); };
    prm.win_mode = ex->window;
    prm.pre_tokens = clampw(ex->pre_tokens);
    prm.next_tokens = clampw(ex->next_tokens);
    prm.amask = ex->atten_mask;
    prm.am_sb = ex->mask_stride_b;
    prm.am_sh = ex->mask_stride_h;
    prm.am_sq = ex->mask_stride_q;
    prm.alibi = ex->alibi;
    prm.pse = static_cast<const uint16_t*>(ex->pse);
    prm.pse_sb = ex->pse_stride_b;
    prm.pse_sh = ex->pse_stride_h;
    prm.pse_sq = ex->pse_stride_q;
    prm.pse_type = ex->pse_type;
    // dropout: keep a byte b when b < keep_prob * 255, as an integer bound
    prm.keep_prob = 1.f;
    prm.keep_thr = 256;
    if (ex->keep_prob > 0.f && ex->keep_prob < 1.f) {
      int thr = 0;
      while (thr < 256 && (double)thr < (double)ex->keep_prob * 255.0) ++thr;
      prm.keep_thr = thr;
      prm.keep_prob = ex->keep_prob;
      prm.drop_key0 = (uint32_t)(ex->seed & 0xFFFFFFFFull);
      prm.drop_key1 = (uint32_t)(ex->seed >> 32);
      prm.drop_ctr0 = ex->offset / 16;
    }
  } else {
    prm.keep_prob = 1.f;
    prm.keep_thr = 256;
  }
  prm.dsq = ds_q;
  prm.dsk = ds_k;
  prm.dsv = ds_v;
  prm.ds_nbq = (Sq + 127) / 128;
  prm.ds_nbk = (Skv + 127) / 128;
  const long long units = (long long)prm.units_per_q * prm.n_qpos;
  if (units > 0x7FFFFFFF) return FA_ERR_SHAPE;

  // Split-KV when the units cannot fill half the GPU: each unit's KV tiles are
  // cut into up to g_max_kv_split pieces of at least two tiles, one CTA each;
  // the pieces leave O / l and the LSE in fp32 scratch and a merge kernel
  // combines them (dense problems only).
  prm.kv_split = 1;
  const int sms = sm_count();
  const int n_kb = (Skv + fa::kBN - 1) / fa::kBN;
  if (!kv_block_idx && !ex && sms > 0 && units * 2 <= sms) {
    int ks = std::min(g_max_kv_split.load(), (int)((sms + units - 1) / units));
    ks = std::min(ks, n_kb / 2);
    if (ks >= 2) prm.kv_split = ks;
  }
  void* parts = nullptr;
  bool parts_owned = false;
  const size_t rows_all = (size_t)B * Hq * Sq;
  if (prm.kv_split > 1) {
    const size_t o_bytes = (size_t)prm.kv_split * rows_all * Dv * 4;
    const size_t bytes = o_bytes + (size_t)prm.kv_split * rows_all * 4;
    if (may_alloc) {
      parts = scratch_alloc(bytes, st);
      parts_owned = parts != nullptr;
    } else if (bytes <= kNoAllocScratchBytes) {
      parts = noalloc_scratch_address();
    }
    if (parts) {
      prm.part_o = static_cast<float*>(parts);
      prm.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(parts) + o_bytes);
    } else {
      prm.kv_split = 1;   // no scratch: run unsplit
    }
  }
  const int grid = (int)std::min<long long>(units * prm.kv_split, 0x7FFFFFFF);
  int rc = ex ? launch_tiled_variant<false, true>(prm, grid, st, D, fp16, conv)
           : prm.kv_split > 1 ? launch_tiled_variant<true>(prm, grid, st, D, fp16, conv)
                              : launch_tiled_variant<false>(prm, grid, st, D, fp16, conv);
  if (rc == FA_OK && prm.kv_split > 1) {
    const unsigned blocks = (unsigned)((rows_all + 7) / 8);
    const cudaError_t e =
        fp16 ? launch_dependent(fa_merge_kernel<false>, blocks, 256, 0, st, prm.part_o,
                                prm.part_lse, o, o_lo, lse, (long long)rows_all, Dv, prm.kv_split)
             : launch_dependent(fa_merge_kernel<true>, blocks, 256, 0, st, prm.part_o,
                                prm.part_lse, o, o_lo, lse, (long long)rows_all, Dv, prm.kv_split);
    if (e != cudaSuccess) rc = cuda_fail(e);
  }
  if (parts_owned) cudaFreeAsync(parts, st);
  return rc;
}

// One warp waits, with the kernels' bounded wait, on an mbarrier that nothing
// ever arrives at: the wait gives up after the configured limit and reports
// the timeout in the status word, and the kernel returns.
__global__ void fa_wait_probe_kernel(int* status, long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(fa::smem_u32(&bar), 1);
    abort_flag = 0;
    fa::fence_mbar_init();
  }
  __syncthreads();
  const fa::WaitCtx wc{reinterpret_cast<volatile int*>(&abort_flag), status, timeout_ns};
  (void)fa::wait_bar(fa::smem_u32(&bar), 0, wc);
}

// fa_fwd and fa_fwd_o_lo on validated arguments (o_lo: the residual output or null).
int fwd_impl(const void* q, const void* k, const void* v, void* o, void* o_lo, float* lse, int B,
             int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
             const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
             const fa_topk_t* topk_idx, float rescale_threshold, void* stream) {
  const int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                          kv_block_idx, topk_idx, rescale_threshold);
  if (rc != FA_OK) return rc;
  const bool fp16 = (mask_mode & (FA_DTYPE_FP16 | FA_V_FP16)) != 0;   // V already fp16
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());

  if (!topk_idx)   // a bf16 V is converted inside the tiled kernel
    return run_tiled(q, k, v, o, o_lo, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode,
                     seqlens, kv_block_idx, rescale_threshold, status, st, /*may_alloc=*/true);
  // top-k: an fp16 copy of the bf16 key latent (V is part of it) in
  // stream-ordered scratch, freed on the same stream
  const size_t nv = (size_t)B * Skv * D;
  void* k16 = const_cast<void*>(k);
  if (!fp16) {
    k16 = scratch_alloc(nv * 2, st);
    if (!k16) return cuda_fail(cudaGetLastError());
    const int rcv = convert_v(k, k16, nv, status, st);
    if (rcv != FA_OK) {
      cudaFreeAsync(k16, st);
      return rcv;
    }
  }
  struct ScratchGuard {
    void* ptr;
    cudaStream_t st;
    ~ScratchGuard() {
      if (ptr) cudaFreeAsync(ptr, st);
    }
  } guard{fp16 ? nullptr : k16, st};
  return run_topk(q, k16, o, o_lo, lse, B, Hq, Sq, Skv, scale, mask_mode, seqlens, topk_idx,
                  rescale_threshold, status, st);
}

// ------------------------------------------------------------------ backward
// S and dP of one batch of the backward's GEMMs are held in fp32; a batch
// covers as many KV planes as fit in this many bytes (at least one).
constexpr size_t kBwdGemmBytes = size_t(1) << 30;
// Query rows per block of the causal backward's GEMMs (each block against the
// keys up to its last row).
constexpr int kBwdRowBlock = 512;

// One cuBLAS handle per device, created on first use: no reduced-precision
// reductions inside the products and no workspace, so that calls on
// different streams share nothing on the device.  The mutex covers a whole
// call's enqueue (the handle's stream is set per call).
std::mutex g_blas_mu;
cublasHandle_t blas_handle() {
  static cublasHandle_t hs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!hs[dev]) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    if (cublasSetMathMode(h, cublasMath_t(CUBLAS_DEFAULT_MATH |
                                          CUBLAS_MATH_DISALLOW_REDUCED_PRECISION_REDUCTION)) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasSetWorkspace(h, nullptr, 0) != CUBLAS_STATUS_SUCCESS) {
      cublasDestroy(h);
      return nullptr;
    }
    hs[dev] = h;
  }
  return hs[dev];
}

// Row-major C[M, N] = alpha op(A) op(B) + beta C over `batch` strided
// matrices (leading dimensions and strides in elements), as the column-major
// product C^T = op(B)^T op(A)^T: A and B bf16 (or fp16) on the tensor cores,
// products exact in fp32, C fp32.
bool gemm_rm16(cublasHandle_t h, cudaDataType_t t, bool ta, bool tb, int M, int N, int K,
               float alpha, const uint16_t* A, int lda, long long sA, const uint16_t* Bm, int ldb,
               long long sB, float beta, float* C, int ldc, long long sC, int batch) {
  return cublasGemmStridedBatchedEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N,
                                    N, M, K, &alpha, Bm, t, ldb, sB, A, t, lda, sA, &beta, C,
                                    CUDA_R_32F, ldc, sC, batch, CUBLAS_COMPUTE_32F,
                                    CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* o_lo,
             const float* lse, const void* dout, void* dq, void* dk, void* dv, int B, int Hq,
             int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
             const int32_t* seqlens, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_NULL;
  if (mask_mode & ~(0xF | FA_DTYPE_FP16)) return FA_ERR_SHAPE;
  const int mask = mask_mode & 0xF;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0 || Dv <= 0 || Hq % Hkv)
    return FA_ERR_SHAPE;
  if (mask > FA_MASK_CAUSAL || !std::isfinite(scale)) return FA_ERR_SHAPE;
  if ((long long)B * Hq > (1LL << 30) || (long long)Sq * 128 > (1LL << 31) ||
      (long long)Skv * 128 > (1LL << 31))
    return FA_ERR_SHAPE;
  if (((long long)B * Hq * Sq + 7) / 8 > 0x7FFFFFFF) return FA_ERR_SHAPE;   // the d_row launch's grid
  if (D != Dv || (D != 64 && D != 128)) return FA_ERR_UNSUPPORTED;
  for (const void* t : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned(t, 16)) return FA_ERR_ALIGN;
  if ((o_lo && !aligned(o_lo, 16)) || !aligned(lse, 4) || (seqlens && !aligned(seqlens, 4)))
    return FA_ERR_ALIGN;
  const bool fp16 = (mask_mode & FA_DTYPE_FP16) != 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  std::lock_guard<std::mutex> lock(g_blas_mu);
  cublasHandle_t h = blas_handle();
  if (!h || cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cuda_fail(cudaErrorUnknown);

  // S and dP straight from the inputs on the tensor cores; P and dS as hi +
  // lo pairs of the inputs' type (about 16 significant bits for bf16, 22 for
  // fp16, whose lo parts reach the subnormals below 2^-14), written in place
  // over S and dP, for dV, dQ and dK; dQ, dK, dV accumulate in fp32.  An fp16
  // dS beyond 65504 sets the range bit of the status word.
  const cudaDataType_t t16 = fp16 ? CUDA_R_16F : CUDA_R_16BF;

  // Stream-ordered scratch: d_row; fp32 dQ; fp32 dK2 and dV2 (two rows per
  // key: its hi and lo parts); K2 (every row of K twice); S and dP of one
  // batch of KV planes in fp32 (then the P and dS pairs).
  const int G = Hq / Hkv;
  const int planes = B * Hkv;
  const size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Skv * D;
  const size_t rows = (size_t)B * Hq * Sq;
  const size_t plane_mat = (size_t)Sq * Skv;
  const int chunk = (int)std::min<size_t>(
      {(size_t)planes, (size_t)65535, std::max<size_t>(1, kBwdGemmBytes / (plane_mat * 8))});
  auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_row = al(rows * 4), b_q = al(nq * 4), b_k2 = al(2 * nk * 4), b_kk = al(2 * nk * 2);
  const size_t b_m = al((size_t)chunk * plane_mat * 4);
  const size_t bytes = b_row + b_q + 2 * b_k2 + b_kk + 2 * b_m;
  uint8_t* scratch = static_cast<uint8_t*>(scratch_alloc(bytes, st));
  if (!scratch) return cuda_fail(cudaGetLastError());
  uint8_t* c = scratch;
  float* d_row = reinterpret_cast<float*>(c);
  c += b_row;
  float* dq32 = reinterpret_cast<float*>(c);
  c += b_q;
  float* dk2 = reinterpret_cast<float*>(c);
  float* dv2 = reinterpret_cast<float*>(c + b_k2);
  c += 2 * b_k2;
  uint16_t* k2 = reinterpret_cast<uint16_t*>(c);
  c += b_kk;
  float* sm = reinterpret_cast<float*>(c);
  float* dpm = reinterpret_cast<float*>(c + b_m);

  int rc = FA_OK;
  auto launched = [&]() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess && rc == FA_OK) rc = cuda_fail(e);
    return rc == FA_OK;
  };
  // every row is a multiple of 8 elements (D = 64 or 128)
  auto grid8 = [](size_t n8) { return (unsigned)std::min<size_t>((n8 + 255) / 256, 4096); };
  auto from32 = [&](const float* in, void* out, size_t n) {
    const size_t n8 = n / 8;
    const auto* i4 = reinterpret_cast<const float4*>(in);
    auto* o4 = static_cast<uint4*>(out);
    if (fp16) fa::fa_bwd_from_f32_kernel<false><<<grid8(n8), 256, 0, st>>>(i4, o4, n8);
    else fa::fa_bwd_from_f32_kernel<true><<<grid8(n8), 256, 0, st>>>(i4, o4, n8);
    return launched();
  };
  auto from32_pairs = [&](const float* in, void* out, size_t n) {   // n output elements
    const size_t n8 = n / 8;
    const auto* i4 = reinterpret_cast<const float4*>(in);
    auto* o4 = static_cast<uint4*>(out);
    if (fp16) fa::fa_bwd_from_f32_pairs_kernel<false><<<grid8(n8), 256, 0, st>>>(i4, o4, n8, D);
    else fa::fa_bwd_from_f32_pairs_kernel<true><<<grid8(n8), 256, 0, st>>>(i4, o4, n8, D);
    return launched();
  };
  bool ok = true;
  {
    const cudaError_t e1 = cudaMemsetAsync(dk2, 0, 2 * nk * 4, st);
    const cudaError_t e2 = e1 == cudaSuccess ? cudaMemsetAsync(dv2, 0, 2 * nk * 4, st) : e1;
    if (e2 != cudaSuccess) {
      rc = cuda_fail(e2);
      ok = false;
    }
  }
  if (ok) {
    fa::fa_bwd_dup_rows_kernel<<<grid8(nk / 8), 256, 0, st>>>(static_cast<const uint4*>(k),
                                                              reinterpret_cast<uint4*>(k2), nk / 8, D);
    ok = launched();
  }
  if (ok) {
    // d_row = rowsum(dO * (O + o_lo)) from the forward's output as given
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    const auto* o16 = static_cast<const uint16_t*>(o);
    const auto* lo16 = static_cast<const uint16_t*>(o_lo);
    const auto* d16 = static_cast<const uint16_t*>(dout);
    if (fp16) fa::fa_bwd_drow_kernel<false><<<blocks, 256, 0, st>>>(o16, lo16, d16, d_row, (long long)rows, D);
    else fa::fa_bwd_drow_kernel<true><<<blocks, 256, 0, st>>>(o16, lo16, d16, d_row, (long long)rows, D);
    ok = launched();
  }
  // per head g of every group and batch of KV planes [p0, p0 + np): the query
  // planes are p * G + g, so Q, dO and dQ advance by G planes per KV plane
  const long long sQ = (long long)G * Sq * D, sK = (long long)Skv * D, sM = (long long)plane_mat;
  const long long sK2 = 2 * sK, sM2 = 2 * sM;   // K2, dK2, dV2; the pairs as 16-bit matrices
  const auto* q16 = static_cast<const uint16_t*>(q);
  const auto* k16 = static_cast<const uint16_t*>(k);
  const auto* v16 = static_cast<const uint16_t*>(v);
  const auto* do16 = static_cast<const uint16_t*>(dout);
  const auto* p2 = reinterpret_cast<const uint16_t*>(sm);    // P pairs: [Sq x 2 Skv] per plane
  const auto* ds2 = reinterpret_cast<const uint16_t*>(dpm);  // dS pairs
  for (int g = 0; ok && g < G; ++g) {
    for (int p0 = 0; ok && p0 < planes; p0 += chunk) {
      const int np = std::min(chunk, planes - p0);
      const long long qo = ((long long)p0 * G + g) * Sq * D, ko = (long long)p0 * sK;
      const long long ko2 = 2 * ko;
      // Causal problems go in blocks of kBwdRowBlock query rows, each against
      // the keys up to its last row only (top-left: row i sees keys j <= i), so
      // that the masked half of S is neither computed nor stored.
      const bool causal = mask == FA_MASK_CAUSAL;
      const int rb = causal ? kBwdRowBlock : Sq;
      for (int r0 = 0; ok && r0 < Sq; r0 += rb) {
        const int r1 = std::min(Sq, r0 + rb), nr = r1 - r0;
        const int nc = causal ? std::min(Skv, r1) : Skv;   // keys [0, nc) of these rows
        fa::BwdGemmRows r{lse, d_row, seqlens, Hkv, G, Sq, Skv, causal, scale, p0, g, r0, nc,
                          status};
        const dim3 eg(nr, np);
        const long long qr = qo + (long long)r0 * D;       // the block's rows of Q, dO, dQ
        const long long mr = (long long)r0 * Skv;           // ... of S, dP (fp32 elements)
        const bool vec = Skv % 8 == 0 && nc % 8 == 0;
        ok = gemm_rm16(h, t16, false, true, nr, nc, D, 1.f, q16 + qr, D, sQ, k16 + ko, D, sK, 0.f,
                       sm + mr, Skv, sM, np);                                 // S = Q K^T
        if (ok) ok = gemm_rm16(h, t16, false, true, nr, nc, D, 1.f, do16 + qr, D, sQ, v16 + ko, D,
                               sK, 0.f, dpm + mr, Skv, sM, np);              // dP = dO V^T
        if (ok) {                                                             // P, dS pairs
          if (fp16) {
            if (vec) fa::fa_bwd_p_ds_kernel<false, 8><<<eg, 256, 0, st>>>(sm, dpm, r);
            else fa::fa_bwd_p_ds_kernel<false, 1><<<eg, 256, 0, st>>>(sm, dpm, r);
          } else {
            if (vec) fa::fa_bwd_p_ds_kernel<true, 8><<<eg, 256, 0, st>>>(sm, dpm, r);
            else fa::fa_bwd_p_ds_kernel<true, 1><<<eg, 256, 0, st>>>(sm, dpm, r);
          }
          ok = launched();
        }
        if (ok) ok = gemm_rm16(h, t16, true, false, 2 * nc, D, nr, 1.f, p2 + 2 * mr, 2 * Skv, sM2,
                               do16 + qr, D, sQ, 1.f, dv2 + ko2, D, sK2, np);  // dV2 += P2^T dO
        if (ok) ok = gemm_rm16(h, t16, false, false, nr, D, 2 * nc, scale, ds2 + 2 * mr, 2 * Skv,
                               sM2, k2 + ko2, D, sK2, 0.f, dq32 + qr, D, sQ, np);  // dQ = scale dS2 K2
        if (ok) ok = gemm_rm16(h, t16, true, false, 2 * nc, D, nr, scale, ds2 + 2 * mr, 2 * Skv,
                               sM2, q16 + qr, D, sQ, 1.f, dk2 + ko2, D, sK2, np);  // dK2 += scale dS2^T Q
      }
      if (!ok && rc == FA_OK) rc = cuda_fail(cudaErrorUnknown);
    }
  }
  if (ok) ok = from32(dq32, dq, nq) && from32_pairs(dk2, dk, nk) && from32_pairs(dv2, dv, nk);
  cudaFreeAsync(scratch, st);
  return rc;
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* o_lo,
           const float* lse, const void* dout, void* dq, void* dk, void* dv, int B, int Hq,
           int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
           const int32_t* seqlens, void* stream) {
  return bwd_impl(q, k, v, o, o_lo, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, Dv, scale,
                  mask_mode, seqlens, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
           int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
           const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
           const fa_topk_t* topk_idx, float rescale_threshold, void* stream) {
  return fwd_impl(q, k, v, o, nullptr, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                  kv_block_idx, topk_idx, rescale_threshold, stream);
}

int fa_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
               const int32_t* seqlens, const fa_extras_t* extras, float rescale_threshold,
               void* stream) {
  if (!extras) return FA_ERR_NULL;
  const int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                          nullptr, nullptr, rescale_threshold);
  if (rc != FA_OK) return rc;
  if ((mask_mode & FA_V_FROM_K) || (mask_mode & 0xF) > FA_MASK_CAUSAL) return FA_ERR_SHAPE;
  const int rce = validate_extras(extras, Skv);
  if (rce != FA_OK) return rce;
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  return run_tiled(q, k, v, o, nullptr, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                   nullptr, rescale_threshold, status, reinterpret_cast<cudaStream_t>(stream),
                   /*may_alloc=*/false, extras);
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* d_scale_q,
               const float* d_scale_k, const float* d_scale_v, int fp8_format, void* o, float* lse,
               int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
               const int32_t* seqlens, const fa_extras_t* extras, float rescale_threshold,
               void* stream) {
  if (!d_scale_q || !d_scale_k || !d_scale_v) return FA_ERR_NULL;
  if (fp8_format != FA_FP8_E4M3 && fp8_format != FA_FP8_E5M2) return FA_ERR_SHAPE;
  if (mask_mode & ~0xF) return FA_ERR_SHAPE;     // o is fp16; no other flag applies
  const int mm = mask_mode | FA_DTYPE_FP16;
  // the arguments as the fp16 call will see them (q8, k8, v8 stand in for the copies)
  int rc = validate(q8, k8, v8, o, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mm, seqlens, nullptr,
                    nullptr, rescale_threshold);
  if (rc != FA_OK) return rc;
  if ((mask_mode & 0xF) > FA_MASK_CAUSAL) return FA_ERR_SHAPE;
  if ((Skv + fa::kBN - 1) / fa::kBN > fa::kMaxSel) return FA_ERR_SHAPE;
  if (!aligned(d_scale_q, 4) || !aligned(d_scale_k, 4) || !aligned(d_scale_v, 4))
    return FA_ERR_ALIGN;
  if (extras) {
    const int rce = validate_extras(extras, Skv);
    if (rce != FA_OK) return rce;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  // exact fp16 copies in stream-ordered scratch; the kernel applies the
  // dequant scales (S by d_q d_k, P by d_v)
  const size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Skv * D,
               nv = (size_t)B * Hkv * Skv * Dv;
  uint8_t* scratch = static_cast<uint8_t*>(scratch_alloc((nq + nk + nv) * 2, st));
  if (!scratch) return cuda_fail(cudaGetLastError());
  void* q16 = scratch;
  void* k16 = scratch + nq * 2;
  void* v16 = scratch + (nq + nk) * 2;
  const bool e5m2 = fp8_format == FA_FP8_E5M2;
  rc = fp8_to_fp16(q8, nullptr, q16, (size_t)B * Hq, Sq, D, e5m2, st);
  if (rc == FA_OK) rc = fp8_to_fp16(k8, nullptr, k16, (size_t)B * Hkv, Skv, D, e5m2, st);
  if (rc == FA_OK) rc = fp8_to_fp16(v8, nullptr, v16, (size_t)B * Hkv, Skv, Dv, e5m2, st);
  fa_extras_t none;
  std::memset(&none, 0, sizeof(none));
  if (rc == FA_OK)
    rc = run_tiled(q16, k16, v16, o, nullptr, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mm, seqlens,
                   nullptr, rescale_threshold, status, st, /*may_alloc=*/true,
                   extras ? extras : &none, d_scale_q, d_scale_k, d_scale_v);
  cudaFreeAsync(scratch, st);
  return rc;
}

int fa_fwd_o_lo(const void* q, const void* k, const void* v, void* o, void* o_lo, float* lse,
                int B, int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale,
                int mask_mode, const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
                const fa_topk_t* topk_idx, float rescale_threshold, void* stream) {
  if (!o_lo) return FA_ERR_NULL;
  if (!aligned(o_lo, 16)) return FA_ERR_ALIGN;
  return fwd_impl(q, k, v, o, o_lo, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                  kv_block_idx, topk_idx, rescale_threshold, stream);
}



int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int Sq, int Skv, int D, int Dv, float scale, int mask_mode,
                   const int32_t* seqlens, const fa_block_sparse_t* kv_block_idx,
                   const fa_topk_t* topk_idx, float rescale_threshold, void* stream) {
  const int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                          kv_block_idx, topk_idx, rescale_threshold);
  if (rc != FA_OK) return rc;
  const bool fp16 = (mask_mode & (FA_DTYPE_FP16 | FA_V_FP16)) != 0;   // latent already fp16
  // the latent's size is checked with the other arguments, before any CUDA call
  const size_t nv = (size_t)B * Skv * D;
  if (topk_idx && !fp16 && nv * 2 > kNoAllocScratchBytes) return FA_ERR_SCRATCH;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  if (!topk_idx)   // a bf16 V is converted inside the tiled kernel; split-KV pieces
                   // use the fixed scratch (unsplit when they do not fit)
    return run_tiled(q, k, v, o, nullptr, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode,
                     seqlens, kv_block_idx, rescale_threshold, status, st, /*may_alloc=*/false);
  void* k16 = const_cast<void*>(k);
  if (!fp16) {
    // bf16 key latent -> fp16 into the fixed scratch (every element is
    // overwritten, so nothing needs clearing first)
    k16 = noalloc_scratch_address();
    if (!k16) return FA_ERR_CUDA;
    const int rcv = convert_v(k, k16, nv, status, st);
    if (rcv != FA_OK) return rcv;
  }
  return run_topk(q, k16, o, nullptr, lse, B, Hq, Sq, Skv, scale, mask_mode, seqlens, topk_idx,
                  rescale_threshold, status, st);
}

int fa_convert_v_fp16(const void* v_bf16, void* v_fp16, int64_t n_elems, void* stream) {
  if (!v_bf16 || !v_fp16) return FA_ERR_NULL;
  if (n_elems <= 0 || n_elems % 8) return FA_ERR_SHAPE;
  if (!aligned(v_bf16, 16) || !aligned(v_fp16, 16)) return FA_ERR_ALIGN;
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  return convert_v(v_bf16, v_fp16, (size_t)n_elems, status, reinterpret_cast<cudaStream_t>(stream));
}

int fa_check_status(void* stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  int h = 0;
  e = cudaMemcpyFromSymbol(&h, g_fa_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (h) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (h & fa::kStatusTimeout) return FA_ERR_DEVICE_TIMEOUT;
  if (h & fa::kStatusRange) return FA_ERR_RANGE;
  return FA_OK;
}

void fa_set_wait_timeout_ns(int64_t ns) { g_timeout_ns.store(ns > 0 ? ns : 2000000000LL); }

int fa_set_max_kv_split(int n) {
  if (n < 1 || n > fa::kMaxSplit) return FA_ERR_SHAPE;
  g_max_kv_split.store(n);
  return FA_OK;
}

int fa_wait_probe(void* stream) {
  int* status = status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fa_wait_probe_kernel<<<1, 32, 0, st>>>(status, g_timeout_ns.load());
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid sizes or descriptor fields";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension / mode combination";
    case FA_ERR_ALIGN: return "tensor base address not aligned";
    case FA_ERR_THRESHOLD: return "rescale_threshold outside [0, 15]";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "bounded on-chip wait expired";
    case FA_ERR_RANGE: return "value outside the fp16 range in an fp16 product (bf16 V, top-k Q or latent; fp16 backward dS)";
    case FA_ERR_SCRATCH: return "bf16 key latent larger than the fixed scratch of fa_fwd_noalloc (32 MiB fp16)";
    default: return "unknown error code";
  }
}

int fa_last_cuda_error(void) { return g_last_cuda.load(); }

#ifdef FA_TRACE
// Profiling builds only: device buffer of kTraceCtas x kTraceCap u64 (zeroed
// by the caller) that receives the cycle-stamped events of the first CTAs.
void fa_debug_set_trace(void* buf) { g_trace = static_cast<unsigned long long*>(buf); }
#endif
const char* fa_last_cuda_error_string(void) {
  return cudaGetErrorName(static_cast<cudaError_t>(g_last_cuda.load()));
}

}  // extern "C"
