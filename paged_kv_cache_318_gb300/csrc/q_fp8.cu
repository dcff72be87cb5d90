// FP8 (E4M3) queries: the per-tensor query quantization, and the exact
// 16-bit copy of the query codes for the kernels that take 16-bit queries.
//
// Source: "vllm/v1/attention/backends/flash_attn.py" (git view and the
// v0.9.0.1 docs page), FlashAttentionImpl.forward: with an fp8 cache the
// query, viewed as [num_tokens, num_heads * head_size], is quantized with
// scaled_fp8_quant(query, layer._q_scale) and the attention call gets
// q_descale = layer._q_scale; the FlashInfer backend page, maybe_quant_query
// and get_xqa_bmm1_scale (bmm1 scale = scale * q_scale * k_scale).
//
// A query value reads back as code * q_scale.  Every E4M3 value is exact in
// f16 and in bf16, so the copy holds the codes' values unscaled and the
// kernels that read it get q_scale through the logit scale: the call hands
// them the product k_scale * q_scale in place of k_scale.
#include "pkv_common.cuh"

namespace pkv {

// 16 elements per step: two 16-byte loads of bf16/f16, one 16-byte store of
// codes.  code = RN_satfinite_e4m3(x / scale), the quotient in IEEE float32.
template <typename T>
__global__ void __launch_bounds__(256)
scaled_fp8_quant_kernel(const T* __restrict__ in, int64_t in_st,
                        uint8_t* __restrict__ out, int64_t out_st,
                        int64_t rows, int cols,
                        const float* __restrict__ scale) {
  // an attention kernel queued next as a programmatic dependent may become
  // resident now (it waits for this grid before reading the codes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int per_row = cols / 16;
  const int64_t total = rows * per_row;
  const float sc = *scale;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                   threadIdx.x;
       i < total; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int c = static_cast<int>(i - r * per_row);
    const T* src = in + r * in_st + c * 16;
    uint4 raw[2];
    raw[0] = *reinterpret_cast<const uint4*>(src);
    raw[1] = *reinterpret_cast<const uint4*>(src + 8);
    const T* e = reinterpret_cast<const T*>(raw);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint16_t lo, hi;
      const float x0 = __fdiv_rn(to_f32<T>(e[4 * j + 0]), sc);
      const float x1 = __fdiv_rn(to_f32<T>(e[4 * j + 1]), sc);
      const float x2 = __fdiv_rn(to_f32<T>(e[4 * j + 2]), sc);
      const float x3 = __fdiv_rn(to_f32<T>(e[4 * j + 3]), sc);
      // cvt puts its first operand in the upper byte
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo)
          : "f"(x1), "f"(x0));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi)
          : "f"(x3), "f"(x2));
      w[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    *reinterpret_cast<uint4*>(out + r * out_st + c * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The query codes q8 [total_q, Hq, D] (byte strides q_st, q_sh) as 16-bit
// values in q16 [total_q, Hq, D] (contiguous); block 0 also writes
// kq = k_scale * q_scale.
template <typename T>
__global__ void __launch_bounds__(256)
widen_q_kernel(const uint8_t* __restrict__ q8, int64_t q_st, int64_t q_sh,
               T* __restrict__ q16, int total_q, int Hq, int D,
               const float* __restrict__ k_scale,
               const float* __restrict__ q_scale, float* __restrict__ kq) {
  // a kernel queued next as a programmatic dependent may become resident
  // now (it waits for this grid before reading the copy)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0 && threadIdx.x == 0) *kq = *k_scale * *q_scale;
  const int per_head = D / 16;
  const int64_t total = static_cast<int64_t>(total_q) * Hq * per_head;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                   threadIdx.x;
       i < total; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t th = i / per_head;
    const int c = static_cast<int>(i - th * per_head);
    const int64_t t = th / Hq;
    const int h = static_cast<int>(th - t * Hq);
    const uint4 raw =
        *reinterpret_cast<const uint4*>(q8 + t * q_st + h * q_sh + c * 16);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t f2;
        const uint16_t codes =
            static_cast<uint16_t>(hh ? (w[j] >> 16) : (w[j] & 0xFFFF));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"(codes));
        const __half2 v = *reinterpret_cast<const __half2*>(&f2);
        o[2 * j + hh] = pack2<T>(__low2float(v), __high2float(v));
      }
    }
    T* dst = q16 + th * D + c * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

namespace {
unsigned grid_for(int64_t total) {
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(current_sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks > 0 ? blocks : 1);
}
}  // namespace

cudaError_t launch_scaled_fp8_quant(const void* in, int64_t in_st, void* out,
                                    int64_t out_st, int64_t rows, int cols,
                                    const float* scale, bool bf16,
                                    cudaStream_t stream) {
  const int64_t total = rows * (cols / 16);
  if (total == 0) return cudaSuccess;
  note_launch();
  const unsigned grid = grid_for(total);
  uint8_t* o = static_cast<uint8_t*>(out);
  if (bf16)
    scaled_fp8_quant_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(in), in_st, o, out_st, rows, cols,
        scale);
  else
    scaled_fp8_quant_kernel<__half><<<grid, 256, 0, stream>>>(
        static_cast<const __half*>(in), in_st, o, out_st, rows, cols, scale);
  return cudaGetLastError();
}

cudaError_t launch_widen_q(const void* q8, int64_t q_st, int64_t q_sh,
                           void* q16, int total_q, int Hq, int D,
                           const float* k_scale, const float* q_scale,
                           float* kq, bool bf16, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(total_q) * Hq * (D / 16);
  note_launch();
  const unsigned grid = grid_for(total);
  const uint8_t* src = static_cast<const uint8_t*>(q8);
  if (bf16)
    widen_q_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        src, q_st, q_sh, static_cast<__nv_bfloat16*>(q16), total_q, Hq, D,
        k_scale, q_scale, kq);
  else
    widen_q_kernel<__half><<<grid, 256, 0, stream>>>(
        src, q_st, q_sh, static_cast<__half*>(q16), total_q, Hq, D, k_scale,
        q_scale, kq);
  return cudaGetLastError();
}

}  // namespace pkv
