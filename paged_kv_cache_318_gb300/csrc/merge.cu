// merge_attn_states: combine two partial attentions by their LSEs.
//
// Source: "vllm/v1/attention/backends/flash_attn.py", cascade_attention and
// _forward_with_dcp (merge_attn_states(output, prefix_output, prefix_lse,
// suffix_output, suffix_lse)); natural-log LSEs as on the FlashInfer backend
// page, which converts its base-2 LSE before this merge.
//
// Elementwise and bandwidth-bound: one thread per 8 consecutive elements of a
// (token, head) row, so every load and store is one 16-byte (or 32-byte for
// fp32) access and a warp touches 32 consecutive chunks.
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

template <typename T>
struct Pack8 {
  __device__ __forceinline__ static void load(const void* base, int64_t idx,
                                              float* v) {
    const uint4 raw = *reinterpret_cast<const uint4*>(
        static_cast<const T*>(base) + idx);
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = to_f32<T>(e[i]);
  }
  __device__ __forceinline__ static void store(void* base, int64_t idx,
                                               const float* v) {
    uint4 raw;
    T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = from_f32<T>(v[i]);
    *reinterpret_cast<uint4*>(static_cast<T*>(base) + idx) = raw;
  }
};
template <>
struct Pack8<float> {
  __device__ __forceinline__ static void load(const void* base, int64_t idx,
                                              float* v) {
    const float4* src =
        reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = src[0], b = src[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ __forceinline__ static void store(void* base, int64_t idx,
                                               const float* v) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

template <typename TO, typename TI>
__global__ void __launch_bounds__(256)
merge_kernel(void* __restrict__ out, const void* __restrict__ o1,
             const float* __restrict__ l1, const void* __restrict__ o2,
             const float* __restrict__ l2, float* __restrict__ lse_out, int T,
             int H, int D) {
  // launched as a programmatic dependent of the kernel before it: its
  // outputs are complete and visible after this (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int chunks = D / 8;
  const int64_t total = static_cast<int64_t>(T) * H * chunks;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                     threadIdx.x;
       idx < total; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / chunks;             // t * H + h
    const int c = static_cast<int>(idx - row * chunks);
    const int t = static_cast<int>(row / H);
    const int h = static_cast<int>(row - static_cast<int64_t>(t) * H);
    const float a = l1[static_cast<int64_t>(h) * T + t];
    const float b = l2[static_cast<int64_t>(h) * T + t];
    // (fmaxf would drop a NaN: a NaN LSE makes a NaN row instead)
    const bool nan_in = isnan(a) || isnan(b);
    const bool pa = a == INFINITY, pb = b == INFINITY;
    const float m = fmaxf(a, b);
    const bool finite = m != -INFINITY && m != INFINITY && !nan_in;
    const float base = finite ? m : 0.f;
    float wa, wb;
    if (pa || pb) {
      // a side with LSE +inf takes all the weight (the formula's limit)
      wa = pa ? 1.f : 0.f;
      wb = pb ? 1.f : 0.f;
    } else {
      wa = (a == -INFINITY || !finite) ? 0.f : __expf(a - base);
      wb = (b == -INFINITY || !finite) ? 0.f : __expf(b - base);
    }
    const float tot = wa + wb;
    const float inv = nan_in ? __int_as_float(0x7fc00000)
                             : (tot > 0.f ? 1.f / tot : 0.f);
    const int64_t e = row * D + c * 8;
    float va[8], vb[8], r[8];
    Pack8<TI>::load(o1, e, va);
    Pack8<TI>::load(o2, e, vb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // a side with zero weight contributes exactly nothing (even if NaN)
      const float x = (wa != 0.f ? wa * va[i] : 0.f) +
                      (wb != 0.f ? wb * vb[i] : 0.f);
      r[i] = x * inv;
    }
    Pack8<TO>::store(out, e, r);
    if (lse_out && c == 0)
      lse_out[static_cast<int64_t>(h) * T + t] =
          nan_in ? __int_as_float(0x7fc00000)
                 : ((pa || pb) ? INFINITY
                               : (tot > 0.f ? base + __logf(tot) : -INFINITY));
  }
}

template <typename TO, typename TI>
static void launch_typed(void* out, const void* o1, const float* l1,
                         const void* o2, const float* l2, float* lse, int T,
                         int H, int D, cudaStream_t stream, bool pdl) {
  const int64_t total = static_cast<int64_t>(T) * H * (D / 8);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(current_sm_count()) * 32;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  note_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  (void)cudaLaunchKernelEx(&cfg, merge_kernel<TO, TI>, out, o1, l1, o2, l2,
                           lse, T, H, D);
}

cudaError_t launch_merge(void* out, const void* o1, const float* l1,
                         const void* o2, const float* l2, float* lse_out,
                         int T, int H, int D, pkv_dtype out_dt,
                         pkv_dtype in_dt, cudaStream_t s, bool pdl) {
#define PKV_MERGE_CASE(OD, ID, TO, TI)                                    \
  if (out_dt == OD && in_dt == ID) {                                      \
    launch_typed<TO, TI>(out, o1, l1, o2, l2, lse_out, T, H, D, s, pdl);  \
    return cudaGetLastError();                                            \
  }
  PKV_MERGE_CASE(PKV_BF16, PKV_BF16, __nv_bfloat16, __nv_bfloat16)
  PKV_MERGE_CASE(PKV_F16, PKV_F16, __half, __half)
  PKV_MERGE_CASE(PKV_F32, PKV_F32, float, float)
  PKV_MERGE_CASE(PKV_BF16, PKV_F32, __nv_bfloat16, float)
  PKV_MERGE_CASE(PKV_F16, PKV_F32, __half, float)
  PKV_MERGE_CASE(PKV_F32, PKV_BF16, float, __nv_bfloat16)
  PKV_MERGE_CASE(PKV_F32, PKV_F16, float, __half)
#undef PKV_MERGE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
