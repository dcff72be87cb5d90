// reshape_and_cache: scatter new K/V rows into the paged cache.
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (reshape_and_cache_flash; the token count is len(slot_mapping));
// v0.9.0.1 docs, FlashAttentionMetadataBuilder.build (padding slots = -1).
//
// Pure data movement: every 16-byte chunk of a (token, kv-head) row of K and
// of V is read once and written once.  One thread moves one chunk of K and
// the matching chunk of V, so a warp covers 512 contiguous bytes of the key
// row and 512 of the value row; the destination rows of one (slot, head) are
// contiguous too (head_size * 2 bytes).  The grid is a flat range over
// (token, head, chunk) so the copy is independent of the cache layout.
#include "pkv_common.cuh"

namespace pkv {

template <int VEC_BYTES>
struct alignas(VEC_BYTES) Vec {
  unsigned char b[VEC_BYTES];
};

template <int VEC_BYTES>
__global__ void __launch_bounds__(256)
cache_write_kernel(const unsigned char* __restrict__ key,
                   const unsigned char* __restrict__ value, int64_t k_st,
                   int64_t k_sh, int64_t v_st, int64_t v_sh,
                   unsigned char* __restrict__ kc,
                   unsigned char* __restrict__ vc, int64_t c_sb, int64_t c_sr,
                   int64_t c_sh, const int64_t* __restrict__ slots,
                   int64_t num_tokens, int Hkv, int row_bytes, int BS,
                   int64_t num_slots, int elem_bytes, unsigned* err) {
  using V = Vec<VEC_BYTES>;
  const int chunks = row_bytes / VEC_BYTES;
  const int64_t per_token = static_cast<int64_t>(Hkv) * chunks;
  const int64_t total = num_tokens * per_token;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                     threadIdx.x;
       idx < total; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_token;
    const int rem = static_cast<int>(idx - t * per_token);
    const int h = rem / chunks;
    const int c = rem - h * chunks;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;                          // padding slot
    if (s >= num_slots) {                         // outside the cache: skip
      if (c == 0 && h == 0) atomicOr(err, kErrBadSlot);
      continue;
    }
    const int64_t blk = s / BS;
    const int64_t off = s - blk * BS;
    const int64_t dst = (blk * c_sb + off * c_sr + h * c_sh) * elem_bytes +
                        static_cast<int64_t>(c) * VEC_BYTES;
    const V kv = *reinterpret_cast<const V*>(
        key + (t * k_st + h * k_sh) * elem_bytes + c * VEC_BYTES);
    const V vv = *reinterpret_cast<const V*>(
        value + (t * v_st + h * v_sh) * elem_bytes + c * VEC_BYTES);
    *reinterpret_cast<V*>(kc + dst) = kv;
    *reinterpret_cast<V*>(vc + dst) = vv;
  }
}

// FP8 (E4M3) cache: each thread quantizes 8 consecutive elements (16 bytes
// of bf16/f16 in, 8 bytes out): code = RN_satfinite_e4m3(x / scale), the
// quotient in IEEE float32.
template <typename T>
__global__ void __launch_bounds__(256)
cache_write_fp8_kernel(const T* __restrict__ key, const T* __restrict__ value,
                       int64_t k_st, int64_t k_sh, int64_t v_st, int64_t v_sh,
                       uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                       int64_t c_sb, int64_t c_sr, int64_t c_sh,
                       const int64_t* __restrict__ slots, int64_t num_tokens,
                       int Hkv, int D, int BS, int64_t num_slots,
                       const float* __restrict__ k_scale,
                       const float* __restrict__ v_scale, unsigned* err) {
  const int chunks = D / 8;
  const int64_t per_token = static_cast<int64_t>(Hkv) * chunks;
  const int64_t total = num_tokens * per_token;
  const float ks = *k_scale, vs = *v_scale;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) +
                     threadIdx.x;
       idx < total; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_token;
    const int rem = static_cast<int>(idx - t * per_token);
    const int h = rem / chunks;
    const int c = rem - h * chunks;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (c == 0 && h == 0) atomicOr(err, kErrBadSlot);
      continue;
    }
    const int64_t blk = s / BS;
    const int64_t off = s - blk * BS;
    const int64_t dst = blk * c_sb + off * c_sr + h * c_sh + c * 8;
#pragma unroll
    for (int mat = 0; mat < 2; ++mat) {
      const T* src = mat ? value + t * v_st + h * v_sh + c * 8
                         : key + t * k_st + h * k_sh + c * 8;
      const float sc = mat ? vs : ks;
      const uint4 raw = *reinterpret_cast<const uint4*>(src);
      const T* e = reinterpret_cast<const T*>(&raw);
      uint32_t packed[2];
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        uint16_t lo, hi;
        const float x0 = __fdiv_rn(to_f32<T>(e[4 * w + 0]), sc);
        const float x1 = __fdiv_rn(to_f32<T>(e[4 * w + 1]), sc);
        const float x2 = __fdiv_rn(to_f32<T>(e[4 * w + 2]), sc);
        const float x3 = __fdiv_rn(to_f32<T>(e[4 * w + 3]), sc);
        // cvt puts its first operand in the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo)
            : "f"(x1), "f"(x0));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi)
            : "f"(x3), "f"(x2));
        packed[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      uint8_t* d = (mat ? vc : kc) + dst;
      *reinterpret_cast<uint2*>(d) = make_uint2(packed[0], packed[1]);
    }
  }
}

cudaError_t launch_cache_write_fp8(const void* key, const void* value,
                                   int64_t k_st, int64_t k_sh, int64_t v_st,
                                   int64_t v_sh, void* kc, void* vc,
                                   const int64_t* cs, const int64_t* slots,
                                   int64_t num_tokens, int Hkv, int D, int BS,
                                   int64_t num_blocks, bool bf16,
                                   const float* k_scale, const float* v_scale,
                                   unsigned* err, cudaStream_t stream) {
  const int64_t total = num_tokens * Hkv * (D / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(current_sm_count()) * 64;
  if (blocks > cap) blocks = cap;
  note_launch();
  if (bf16)
    cache_write_fp8_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256,
                                            0, stream>>>(
        static_cast<const __nv_bfloat16*>(key),
        static_cast<const __nv_bfloat16*>(value), k_st, k_sh, v_st, v_sh,
        static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), cs[0], cs[1],
        cs[2], slots, num_tokens, Hkv, D, BS, num_blocks * BS, k_scale,
        v_scale, err);
  else
    cache_write_fp8_kernel<__half><<<static_cast<unsigned>(blocks), 256, 0,
                                     stream>>>(
        static_cast<const __half*>(key), static_cast<const __half*>(value),
        k_st, k_sh, v_st, v_sh, static_cast<uint8_t*>(kc),
        static_cast<uint8_t*>(vc), cs[0], cs[1], cs[2], slots, num_tokens, Hkv,
        D, BS, num_blocks * BS, k_scale, v_scale, err);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const void* key, const void* value,
                               int64_t k_st, int64_t k_sh, int64_t v_st,
                               int64_t v_sh, void* kc, void* vc,
                               const int64_t* cs, const int64_t* slots,
                               int64_t num_tokens, int Hkv, int D, int BS,
                               int64_t num_blocks, int elem_bytes,
                               unsigned* err, cudaStream_t stream) {
  const int row_bytes = D * elem_bytes;
  // 16-byte chunks when every row start is 16-byte aligned, else 2 bytes.
  auto aligned16 = [&](const void* p, int64_t a, int64_t b) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
           ((a * elem_bytes) % 16 == 0) && ((b * elem_bytes) % 16 == 0);
  };
  const bool vec16 = row_bytes % 16 == 0 && aligned16(key, k_st, k_sh) &&
                     aligned16(value, v_st, v_sh) &&
                     aligned16(kc, cs[0], cs[1]) &&
                     aligned16(vc, cs[0], cs[1]) &&
                     (cs[2] * elem_bytes) % 16 == 0;
  const int vec = vec16 ? 16 : 2;
  const int64_t total = num_tokens * Hkv * (row_bytes / vec);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(current_sm_count()) * 64;
  if (blocks > cap) blocks = cap;   // grid-stride beyond
  const int64_t num_slots = num_blocks * BS;
  note_launch();
  if (vec16) {
    cache_write_kernel<16><<<static_cast<unsigned>(blocks), threads, 0,
                             stream>>>(
        static_cast<const unsigned char*>(key),
        static_cast<const unsigned char*>(value), k_st, k_sh, v_st, v_sh,
        static_cast<unsigned char*>(kc), static_cast<unsigned char*>(vc),
        cs[0], cs[1], cs[2], slots, num_tokens, Hkv, row_bytes, BS, num_slots,
        elem_bytes, err);
  } else {
    cache_write_kernel<2><<<static_cast<unsigned>(blocks), threads, 0,
                            stream>>>(
        static_cast<const unsigned char*>(key),
        static_cast<const unsigned char*>(value), k_st, k_sh, v_st, v_sh,
        static_cast<unsigned char*>(kc), static_cast<unsigned char*>(vc),
        cs[0], cs[1], cs[2], slots, num_tokens, Hkv, row_bytes, BS, num_slots,
        elem_bytes, err);
  }
  return cudaGetLastError();
}

}  // namespace pkv
