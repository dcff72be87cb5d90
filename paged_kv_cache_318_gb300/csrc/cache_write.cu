// reshape_and_cache: scatter new K/V rows into the paged cache.
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (reshape_and_cache_flash; the token count is len(slot_mapping));
// v0.9.0.1 docs, FlashAttentionMetadataBuilder.build (padding slots = -1).
//
// Pure data movement: every 16-byte chunk of a (token, kv-head) row of K and
// of V is read once and written once.  Rows of 64, 128 or 256 16-bit
// elements go through cache_write_warp_kernel (a warp per token); other row
// sizes or alignments through cache_write_kernel, one thread per chunk of K
// and the matching chunk of V over a flat range of (token, head, chunk), so
// the copy is independent of the cache layout.
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

// The same copy with one warp per token, for rows of CH 16-byte chunks (CH
// = 8, 16 or 32: head sizes 64, 128, 256 in 16 bits) and Hkv * CH <= 32 *
// UNROLL.  The token's slot and its (block, offset) are resolved once per
// warp; lane l moves chunks l, l + 32, ... of the token's K and V rows
// (UNROLL of each in flight), whose (head, chunk) offsets it computes once.
// The per-chunk kernel above spends most of its issue slots on the 64-bit
// divisions of its index math (measured on GB300: 69 % issue-active at
// 0.56 of the HBM peak).
template <int CH, int UNROLL>
__global__ void __launch_bounds__(256)
cache_write_warp_kernel(const unsigned char* __restrict__ key,
                        const unsigned char* __restrict__ value, int64_t k_st,
                        int64_t k_sh, int64_t v_st, int64_t v_sh,
                        unsigned char* __restrict__ kc,
                        unsigned char* __restrict__ vc, int64_t c_sb,
                        int64_t c_sr, int64_t c_sh,
                        const int64_t* __restrict__ slots, int64_t num_tokens,
                        int Hkv, int BS, int bs_shift, int64_t num_slots,
                        int elem_bytes, unsigned* err) {
  // an attention kernel queued next as a programmatic dependent may become
  // resident now (it waits for this grid before reading the cache)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using V = uint4;    // (16 bytes in four 32-bit registers)
  constexpr int LOG_CH = CH == 8 ? 3 : (CH == 16 ? 4 : 5);
  const int lane = threadIdx.x & 31;
  const int64_t warp0 =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int per_token = Hkv * CH;
  int64_t ko[UNROLL], vo[UNROLL], co[UNROLL];
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) {
    const int j = u * 32 + lane;
    const int h = j >> LOG_CH, c = j & (CH - 1);
    ko[u] = (h * k_sh) * elem_bytes + c * 16;
    vo[u] = (h * v_sh) * elem_bytes + c * 16;
    co[u] = (h * c_sh) * elem_bytes + c * 16;
  }
#pragma unroll 1
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;                          // padding slot
    if (s >= num_slots) {                         // outside the cache: skip
      if (lane == 0) atomicOr(err, kErrBadSlot);
      continue;
    }
    const int64_t blk = bs_shift >= 0 ? (s >> bs_shift) : s / BS;
    const int64_t off = s - blk * BS;
    const unsigned char* ks = key + t * k_st * elem_bytes;
    const unsigned char* vs = value + t * v_st * elem_bytes;
    const int64_t d0 = (blk * c_sb + off * c_sr) * elem_bytes;
    V kb[UNROLL], vb[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (u * 32 + lane < per_token) {
        kb[u] = *reinterpret_cast<const V*>(ks + ko[u]);
        vb[u] = *reinterpret_cast<const V*>(vs + vo[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (u * 32 + lane < per_token) {
        *reinterpret_cast<V*>(kc + d0 + co[u]) = kb[u];
        *reinterpret_cast<V*>(vc + d0 + co[u]) = vb[u];
      }
    }
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
  const int chunks = row_bytes / 16;
  const int per_token = Hkv * chunks;
  if (vec16 && (chunks == 8 || chunks == 16 || chunks == 32) &&
      per_token <= 256) {
    int bs_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
      if ((1 << sh) == BS) bs_shift = sh;
    int64_t blocks = (num_tokens + 7) / 8;        // 8 warps per block
    const int64_t cap = static_cast<int64_t>(current_sm_count()) * 16;
    if (blocks > cap) blocks = cap;               // grid-stride beyond
    const auto* k8 = static_cast<const unsigned char*>(key);
    const auto* v8 = static_cast<const unsigned char*>(value);
    auto* kc8 = static_cast<unsigned char*>(kc);
    auto* vc8 = static_cast<unsigned char*>(vc);
    const int64_t num_slots = num_blocks * BS;
    note_launch();
    const unsigned g = static_cast<unsigned>(blocks);
    auto go = [&](auto kern) {
      kern<<<g, 256, 0, stream>>>(k8, v8, k_st, k_sh, v_st, v_sh, kc8, vc8,
                                  cs[0], cs[1], cs[2], slots, num_tokens, Hkv,
                                  BS, bs_shift, num_slots, elem_bytes, err);
    };
    const int unroll = per_token <= 32 ? 1 : per_token <= 64 ? 2
                     : per_token <= 128 ? 4 : 8;
#define PKV_CW(CH_)                                                   \
  if (chunks == CH_) {                                                \
    if (unroll == 1) go(cache_write_warp_kernel<CH_, 1>);             \
    else if (unroll == 2) go(cache_write_warp_kernel<CH_, 2>);        \
    else if (unroll == 4) go(cache_write_warp_kernel<CH_, 4>);        \
    else go(cache_write_warp_kernel<CH_, 8>);                         \
  }
    PKV_CW(8) else PKV_CW(16) else PKV_CW(32)
#undef PKV_CW
    return cudaGetLastError();
  }
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
