// Shared device helpers and the internal launch interface of libpkv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Error bits OR-ed into the device error word by kernels that skip an access.
constexpr unsigned kErrBadBlock = 1u;   // block id outside [0, num_blocks)
constexpr unsigned kErrBadSlot = 2u;    // slot outside the cache
constexpr unsigned kErrBadTable = 4u;   // key beyond the block-table row
constexpr unsigned kErrTimeout = 8u;    // a bounded wait gave up
constexpr unsigned kErrSmemAlign = 16u; // shared memory not 1024-byte aligned
constexpr unsigned kErrQueryLen = 32u;  // a request's query count is above
                                        // the max_seqlen_q the call gave

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared async copy; src_bytes == 0 writes zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src,
                                            int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0,
                                            uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0,
                                                  uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a,
                                          uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma_16816<__nv_bfloat16>(float* d,
                                                         const uint32_t* a,
                                                         uint32_t b0,
                                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma_16816<__half>(float* d, const uint32_t* a,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Hardware base-2 exponential and logarithm (MUFU).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) {
  return __half2float(x);
}
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Key range [kmin, kmax) that any query row of tokens [i_first, i_last] of a
// request (q_len queries, L keys) may see.  Query i sits at p = L - q_len + i.
__device__ __forceinline__ void key_range(int L, int q_len, int i_first,
                                          int i_last, int causal, int wl,
                                          int wr, int& kmin, int& kmax) {
  const int ctx = L - q_len;
  const int p_lo = ctx + i_first, p_hi = ctx + i_last;
  kmax = L;
  if (causal) kmax = min(kmax, p_hi + 1);
  if (wr >= 0) kmax = min(kmax, p_hi + wr + 1);
  kmin = 0;
  if (wl >= 0) kmin = max(0, p_lo - wl);
  if (kmax < kmin) kmax = kmin;
}

// Hardware tanh (tanh.approx.f32); its relative error (about 2^-11) keeps
// soft-capped logits well inside the output tolerance.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Split-KV: split s of a request's key range [kmin, kmax) covers `chunk`
// keys (a multiple of 64) counted from kmin rounded down to 64, so every
// split after the first starts on a 64-key boundary.  The last of the
// request's splits (at most max_splits) takes the rest of the range.
__device__ __forceinline__ int split_count(int kmin, int kmax, int chunk,
                                           int max_splits) {
  const int base = kmin & ~63;
  return min(max((kmax - base + chunk - 1) / chunk, 1), max_splits);
}
__device__ __forceinline__ void split_bounds(int kmin, int kmax, int chunk,
                                             int nsplit, int s, int& lo,
                                             int& hi) {
  const int base = kmin & ~63;
  lo = max(kmin, base + s * chunk);
  hi = (s == nsplit - 1) ? kmax : min(kmax, base + (s + 1) * chunk);
  if (hi < lo) hi = lo;
}

// Byte offset of 16-byte chunk `ch` of row `r` in a tile whose rows are
// ROW_BYTES apart, XOR-swizzled over 8-chunk groups (conflict-free ldmatrix).
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return static_cast<uint32_t>(r * ROW_BYTES + ((ch ^ (r & 7)) << 4));
}

// ------------------------------------------------------- internal interface

// Parameters of the block-table attention kernels.
struct AttnParams {
  const void* q;
  int64_t q_st, q_sh;
  const void* kc;
  const void* vc;
  int64_t c_sb, c_sr, c_sh;   // cache strides: block, row-in-block, kv-head
  int rb;                     // TMA kernels: rows per K/V box
  int kv_order_hnd;           // TMA kernels: 1 = head stride > row stride
  void* out;
  int64_t o_st, o_sh;
  float* lse;                 // [Hq, total_q] natural log, or null
  int total_q;
  const int32_t* cu_q;
  const int32_t* seqused_k;
  // non-paged mode: keys of request b are rows cu_k[b] .. cu_k[b+1]-1 of one
  // K/V tensor of total_k rows (c_sr: row stride, c_sh: head stride); null
  // = paged
  const int32_t* cu_k;
  int total_k;
  int batch;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  int64_t num_blocks;
  int Hq, Hkv, G, BS;
  int bs_shift;               // log2(BS) when BS is a power of two, else -1
  float scale;                // softmax scale (natural units)
  float softcap;              // 0 = none
  const float* alibi;         // [Hq] or null
  const float* sinks;         // [Hq] sink logits (natural log) or null
  int kv_fp8;                 // cache holds E4M3 codes (1 byte / element)
  const float* k_scale;       // fp8: device scalar, value = code * scale
  const float* v_scale;
  // E4M3 query codes (1 byte / element, q_st / q_sh in bytes), value =
  // code * (*q_scale); only the persistent decode kernel reads them (the
  // other kernels get a 16-bit copy and k_scale * q_scale as k_scale)
  int q_fp8;
  const float* q_scale;
  // TMA decode kernel launched as a programmatic dependent of the grid
  // before it: a zeroed counter of finished CTAs (null = ordinary launch)
  int* pdl_done;
  int causal, wl, wr;
  // which requests this launch owns: rows = q_b * G in [min_rows, max_rows]
  int min_rows, max_rows;
  // split-KV: keys per split (0 = no split: write out/lse directly)
  int chunk;
  float* part_o;              // [S, part_rows, Hq, D] fp32
  float* part_lse;            // [S, Hq, part_rows] fp32 natural log
  // partial rows: a token's own index (part_tpr = 0, part_rows = total_q)
  // or, compact, part_tpr rows per request (see part_row)
  int part_tpr, part_rows;
  // persistent prefill: one int of workspace the kernel hands work items
  // out through (the launcher zeroes it first); null = fixed item order
  int* sched;
  int sched_zeroed;           // the caller has zeroed *sched already
  // persistent decode: the tile sequence is cut into sk_chunks chunks (one
  // per CTA); per chunk, the unit it starts inside (x) and the unit it
  // starts that runs past its end (y), -1 for none.  Partial slots hold
  // sk_rows rows.
  int2* sk_marks;
  int sk_chunks;
  int sk_rows;
  // persistent prefill split-KV: key splits per work item (1 = none); with
  // more, partials go to pre_o [S, total_q, Hq, D] / pre_lse [S, Hq,
  // total_q] and launch_prefill_split_combine folds them
  int pre_splits;
  float* pre_o;
  float* pre_lse;
  // persistent prefill: at most this many CTAs (0 = one per SM), leaving
  // the other SMs to a kernel running beside it
  int max_ctas;
  unsigned* err;
  // bounded mbarrier waits of the decode kernels give up after this many
  // nanoseconds (pkv_set_wait_limit_ns; the drains at exit keep 2 s)
  uint64_t wait_ns;
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  int part_tpr, part_rows;    // partial row layout (see AttnParams)
  void* out;
  int64_t o_st, o_sh;
  float* lse;
  int total_q;
  const int32_t* cu_q;
  const int32_t* seqused_k;
  const int32_t* cu_k;        // non-paged mode (see AttnParams)
  int batch, Hq, G, D;
  int causal, wl, wr;
  int chunk, splits;
  int min_rows, max_rows;
  const float* sinks;         // [Hq] sink logits or null (added once here)
};

// Row of token tok (request b, first token q0) in the split-KV partial
// buffers: the token itself, or with part_tpr > 0 row (tok - q0) of request
// b's block of part_tpr rows.  Only decode-class requests (at most 16 / G
// tokens) write partials, so the compact form needs batch * 16 / G rows
// instead of total_q.
__device__ __forceinline__ int64_t part_row(int part_tpr, int b, int q0,
                                            int tok) {
  return part_tpr > 0 ? static_cast<int64_t>(b) * part_tpr + (tok - q0)
                      : static_cast<int64_t>(tok);
}

// Final normalisation of one row: acc is relative to the running max m
// (log2 units), l the running sum.  With a sink logit (natural units), it is
// one more term of the denominator.  Returns 1/denominator relative to m in
// *inv and the natural-log LSE.
__device__ __forceinline__ void finish_row(float m, float l, const float* sinks,
                                          int h, float* inv, float* lse) {
  if (!sinks) {
    *inv = l > 0.f ? 1.f / l : 0.f;
    *lse = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
    return;
  }
  const float z = sinks[h] * kLog2e;
  const float M = fmaxf(m, z);
  const float em = ex2(m - M);             // m = -inf -> 0
  const float den = l * em + ex2(z - M);
  *inv = em / den;
  *lse = (M + lg2(den)) * kLn2;
}

// Count one kernel launch (reported by pkv_launch_count).
void note_launch();

// SM count of the current device (looked up once per device; 1 if the
// lookup fails).  Grid-stride kernels size their grids from it.
int current_sm_count();

// Raise the dynamic shared-memory limit of kernel `kern` to `bytes` on the
// current device, once per (kernel, device): the attribute is per device,
// so one process driving several GPUs sets it on each.
cudaError_t smem_opt_in(const void* kern, int bytes);

// Set this thread's pkv_last_error message.
void set_last_error(const char* msg);

// Decode kernel geometry (rows = q_len * G <= kDecodeRows go to it).
constexpr int kDecodeRows = 16;
constexpr int kDecodeKT = 64;     // keys per pipeline tile
// Resident decode CTAs per SM: every decode configuration (both kernels,
// every head size) takes 66-73 KB of shared memory and <= 21K registers.
constexpr int kDecodeCtasPerSm = 3;

cudaError_t launch_cache_write(const void* key, const void* value,
                               int64_t k_st, int64_t k_sh, int64_t v_st,
                               int64_t v_sh, void* kc, void* vc,
                               const int64_t* cs, const int64_t* slots,
                               int64_t num_tokens, int Hkv, int D, int BS,
                               int64_t num_blocks, int elem_bytes,
                               unsigned* err, cudaStream_t stream);

cudaError_t launch_cache_write_fp8(const void* key, const void* value,
                                   int64_t k_st, int64_t k_sh, int64_t v_st,
                                   int64_t v_sh, void* kc, void* vc,
                                   const int64_t* cs, const int64_t* slots,
                                   int64_t num_tokens, int Hkv, int D, int BS,
                                   int64_t num_blocks, bool bf16,
                                   const float* k_scale, const float* v_scale,
                                   unsigned* err, cudaStream_t stream);
cudaError_t launch_fp8_dequant_pages(const AttnParams& p, int D, bool bf16,
                                     void* mock_k, void* mock_v,
                                     int32_t* mock_table, cudaStream_t stream);
// E4M3 queries (q_fp8.cu): the per-tensor quantization, and the exact
// 16-bit copy of the codes plus kq = k_scale * q_scale.
cudaError_t launch_scaled_fp8_quant(const void* in, int64_t in_st, void* out,
                                    int64_t out_st, int64_t rows, int cols,
                                    const float* scale, bool bf16,
                                    cudaStream_t stream);
cudaError_t launch_widen_q(const void* q8, int64_t q_st, int64_t q_sh,
                           void* q16, int total_q, int Hq, int D,
                           const float* k_scale, const float* q_scale,
                           float* kq, bool bf16, cudaStream_t stream);

cudaError_t launch_decode_attn(const AttnParams& p, int D, bool bf16,
                               int grid_x, int grid_y, cudaStream_t stream);
cudaError_t launch_prefill_attn_mma(const AttnParams& p, int D, bool bf16,
                                    int grid_y, cudaStream_t stream);
// *splits_used: the key splits the launch wrote partials for (1 = the
// outputs themselves were written).
// pdl: launch as a programmatic dependent of the kernel queued just before
// (the call's decode kernels, which write other requests' rows).
cudaError_t launch_prefill_attn_tc(const AttnParams& p, int D, bool bf16,
                                   int grid_y, bool p_in_tmem,
                                   int* splits_used, cudaStream_t stream,
                                   bool pdl = false);
// Fold the prefill kernel's split-KV partials (p.splits of them, every one
// written for each row) of the requests with rows >= p.min_rows.
cudaError_t launch_prefill_split_combine(const CombineParams& p,
                                         int max_seqlen_q, bool bf16,
                                         cudaStream_t stream);
int prefill_tc_block_keys(int D);
// Decode attention with TMA page loads (decode_tma.cu); 16-bit caches.
cudaError_t launch_decode_attn_tma(const AttnParams& p, int D, bool bf16,
                                   int grid_x, cudaStream_t stream);

// pdl: launch as a programmatic dependent of the decode grid just queued.
cudaError_t launch_split_combine(const CombineParams& p, bool bf16,
                                 cudaStream_t stream, bool pdl = false);
// Persistent decode attention (decode_sk.cu): 16-bit caches with D in {64,
// 128, 256}, E4M3 caches with D in {128, 256}.  decode_sk_ctas gives the
// launch's CTA count on the current device (resident CTAs per SM x sms);
// the launch needs decode_sk_workspace_bytes(D, ctas, rows) of scratch
// (256-byte aligned) for the pieces of units that chunk boundaries cut,
// rows = the most packed query rows a decode-class request can have
// (min(16, G * max_seqlen_q)).
// q8: E4M3 query codes too (needs kv8).
bool decode_sk_supported(int D, bool kv8);
cudaError_t decode_sk_ctas(int D, bool bf16, bool kv8, bool q8, int sms,
                           int* ctas);
size_t decode_sk_workspace_bytes(int D, int ctas, int rows);
// pdl: launch as a programmatic dependent of the kernel queued before it
// (the kernel waits for it at its start).
cudaError_t launch_decode_attn_sk(const AttnParams& p, int D, bool bf16,
                                  int ctas, int rows, void* scratch,
                                  bool pdl, cudaStream_t stream);
// Required workspace bytes of an attention call (pkv_api.cu): the split-KV
// partials and fp8 copies it needs, not the optional prefill tail.
size_t required_workspace_bytes(int batch, int total_q, int max_seqlen_q,
                                int max_seqlen_k, int num_heads,
                                int num_kv_heads, int head_size,
                                int block_size, int causal, int window_left,
                                int window_right, int num_splits);
// pdl: launch as a programmatic dependent of the kernel queued before it.
cudaError_t launch_merge(void* out, const void* o1, const float* l1,
                         const void* o2, const float* l2, float* lse_out,
                         int T, int H, int D, pkv_dtype out_dt,
                         pkv_dtype in_dt, cudaStream_t stream,
                         bool pdl = false);

// ---- E4M3 caches: codes to f16 in registers (both decode kernels)

// Four E4M3 codes (low byte first) -> two f16x2 (exact).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo,
                                              uint32_t& hi) {
  asm("{\n.reg .b16 a, b;\n"
      "mov.b32 {a, b}, %2;\n"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// An 8-bit 16 x 16 block of shared memory (row addresses from lanes 0-15),
// transposed: lane t receives rows 4 (t % 4) .. + 3 of column t / 4 in d0
// and of column t / 4 + 8 in d1 (row 4 (t % 4) in the low byte).
__device__ __forceinline__ void ldmatrix_b8_trans(uint32_t addr, uint32_t& d0,
                                                  uint32_t& d1) {
  asm volatile(
      "ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];"
      : "=r"(d0), "=r"(d1)
      : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

template <typename T>
__device__ __forceinline__ float elem_f32(uint32_t w, int hi);
template <>
__device__ __forceinline__ float elem_f32<__nv_bfloat16>(uint32_t w,
                                                         int hi) {
  return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}
template <>
__device__ __forceinline__ float elem_f32<__half>(uint32_t w, int hi) {
  return __half2float(__ushort_as_half(
      static_cast<unsigned short>(hi ? (w >> 16) : (w & 0xffffu))));
}

}  // namespace pkv
