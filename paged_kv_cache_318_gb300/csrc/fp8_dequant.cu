// FP8 cache, prefill side: convert the pages a prefill-class request reads
// into a 16-bit scratch cache, so the tensor-core prefill kernels run on it.
// The E4M3 codes convert exactly (no scale applied here); the prefill kernels
// fold k_scale into the logit scale and v_scale into the output, so no
// rounding is added beyond the fp8 quantization itself.
//
// Source: the FlashInfer backend page, _trtllm_prefill_attn_kvfp8_dequant
// (grid over (request, page of the request), written to a contiguous "mock"
// cache with its own block table; that helper multiplies by the scale before
// rounding to 16 bits, this one keeps the codes exact).  Decode-class
// requests keep reading the fp8 cache directly in the decode kernel, where
// the halved bytes matter.
//
// Scratch layout: mock K and V caches [batch * max_blocks, BS, Hkv, D]
// (NHD, contiguous) and a mock block table [batch, max_blocks] whose entry
// (b, j) is page b * max_blocks + j.
#include "pkv_common.cuh"

namespace pkv {

template <typename T>
__global__ void __launch_bounds__(256)
fp8_dequant_pages_kernel(const AttnParams p, T* __restrict__ mock_k,
                         T* __restrict__ mock_v, int32_t* __restrict__ table,
                         int D) {
  // one block per (request, table column) page, grid-stride over them
  const int64_t pages = static_cast<int64_t>(p.batch) * p.max_blocks;
  for (int64_t mpage = blockIdx.x; mpage < pages; mpage += gridDim.x) {
    const int b = static_cast<int>(mpage / p.max_blocks);
    const int j = static_cast<int>(mpage - static_cast<int64_t>(b) *
                                               p.max_blocks);
    if (threadIdx.x == 0) table[mpage] = static_cast<int32_t>(mpage);
    const int q0 = p.cu_q[b];
    const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
    if (q0 < 0 || q_len <= 0 || q_len * p.G < p.min_rows) continue;
    const int L_tab = min(p.seqused_k[b], p.max_blocks * p.BS);
    if (static_cast<int64_t>(j) * p.BS >= L_tab) continue;
    const int blk = p.block_table[static_cast<int64_t>(b) * p.bt_stride + j];
    const bool bad = blk < 0 || blk >= p.num_blocks;
    if (bad && threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
    const int per_row = p.Hkv * (D / 8);
    const unsigned char* K8 = static_cast<const unsigned char*>(p.kc);
    const unsigned char* V8 = static_cast<const unsigned char*>(p.vc);
    for (int e = threadIdx.x; e < p.BS * per_row; e += blockDim.x) {
      const int row = e / per_row;
      const int rem = e - row * per_row;
      const int h = rem / (D / 8), c = rem - h * (D / 8);
      const int64_t dst =
          ((mpage * p.BS + row) * p.Hkv + h) * static_cast<int64_t>(D) + c * 8;
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        uint4 out = make_uint4(0, 0, 0, 0);
        if (!bad) {
          const int64_t src = static_cast<int64_t>(blk) * p.c_sb +
                              static_cast<int64_t>(row) * p.c_sr +
                              static_cast<int64_t>(h) * p.c_sh + c * 8;
          const uint2 raw = *reinterpret_cast<const uint2*>(
              (mat ? V8 : K8) + src);
          const uint32_t w[2] = {raw.x, raw.y};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t f2;
              const uint16_t codes = static_cast<uint16_t>(
                  hh ? (w[q] >> 16) : (w[q] & 0xFFFF));
              asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"(codes));
              const __half2 v = *reinterpret_cast<const __half2*>(&f2);
              o[2 * q + hh] = pack2<T>(__low2float(v), __high2float(v));
            }
          }
          out = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>((mat ? mock_v : mock_k) + dst) = out;
      }
    }
  }
}

cudaError_t launch_fp8_dequant_pages(const AttnParams& p, int D, bool bf16,
                                     void* mock_k, void* mock_v,
                                     int32_t* mock_table,
                                     cudaStream_t stream) {
  const int64_t pages = static_cast<int64_t>(p.batch) * p.max_blocks;
  const int64_t cap = static_cast<int64_t>(current_sm_count()) * 16;
  const unsigned grid =
      static_cast<unsigned>(pages < cap ? (pages > 0 ? pages : 1) : cap);
  note_launch();
  if (bf16)
    fp8_dequant_pages_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        p, static_cast<__nv_bfloat16*>(mock_k),
        static_cast<__nv_bfloat16*>(mock_v), mock_table, D);
  else
    fp8_dequant_pages_kernel<__half><<<grid, 256, 0, stream>>>(
        p, static_cast<__half*>(mock_k), static_cast<__half*>(mock_v),
        mock_table, D);
  return cudaGetLastError();
}

}  // namespace pkv
