// C ABI of libpkv: argument validation, the split plan, and kernel launches.
//
// Every entry point validates its arguments on the host before it enqueues
// anything; invalid calls return a pkv_status and a per-thread message and
// launch nothing.  Kernels never trap: out-of-range indices are skipped and
// recorded in a device error word (pkv_check_device_errors reads it).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "pkv_common.cuh"

namespace pkv {

__device__ unsigned g_device_error = 0;

static std::atomic<uint64_t> g_launches{0};
// prefill kernel: PKV_PREFILL_TCGEN05 or PKV_PREFILL_MMA_SYNC
static std::atomic<int> g_prefill_kernel{PKV_PREFILL_TCGEN05};
// decode kernel: PKV_DECODE_AUTO, PKV_DECODE_PERSISTENT, PKV_DECODE_TMA or
// PKV_DECODE_CP_ASYNC
static std::atomic<int> g_decode_kernel{PKV_DECODE_AUTO};
// limit of the decode kernels' bounded waits (pkv_set_wait_limit_ns)
static std::atomic<uint64_t> g_wait_limit_ns{PKV_WAIT_LIMIT_DEFAULT_NS};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

thread_local std::string g_last_error;

pkv_status fail(pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// Per-device facts, looked up once with that device current.
pkv_status device_info(unsigned** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_err_ptr[dev] = static_cast<unsigned*>(ptr);
    g_sm_count[dev] = n;
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_sm_count[dev];
  return PKV_OK;
}

bool aligned16(const void* p) {
  return reinterpret_cast<uintptr_t>(p) % 16 == 0;
}
bool stride16(int64_t s, int elem) { return (s * elem) % 16 == 0; }

// ----------------------------------------------------------- split plan

// When the decode-class requests run first (on the persistent decode
// kernel), launch the prefill kernel as a programmatic dependent of the
// decode kernels (1) or after them (0): its CTAs then take the SMs the
// decode's static chunks leave early.  Measured on GB300, same box: the
// Gemma-like mixed batch (124 decodes + 4 prefill chunks) 0.8393 against
// 0.8424 ms.  (Calls whose decodes take the per-unit kernel launch the
// prefill kernel first instead.)
#ifndef PKV_PREFILL_AFTER_DECODE_PDL
#define PKV_PREFILL_AFTER_DECODE_PDL 1
#endif

// Units of at least this many keys count as long for the decode kernel
// choice.
constexpr int64_t kLongUnitKeys = 2048;

struct Plan {
  int64_t range = 0;      // widest key range of a decode-class unit
  bool decode = false;    // launch the decode (<= 16 packed rows) kernel
  bool prefill = false;   // launch the prefill kernel
  int splits = 1;         // decode grid.x
  int chunk = 0;          // keys per split; 0 = write outputs directly
  int prefill_tiles = 0;  // prefill grid.y
  // decode partial rows: per token (tpr 0) or tpr rows per request
  int part_tpr = 0, part_rows = 0;
  size_t part_o_bytes = 0, part_lse_bytes = 0;
  size_t workspace = 0;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Plan make_plan(int batch, int total_q, int max_q, int max_k, int Hq, int Hkv,
               int D, int causal, int wl, int wr, int num_splits, int sms,
               int fixed_split = 0) {
  Plan pl;
  const int G = Hq / Hkv;
  if (batch == 0 || max_q == 0) return pl;
  // Every request has at least total_q - (batch - 1) * max_q queries.  When
  // that many rows exceed the decode kernel's, no request is decode-class:
  // the decode kernel is not launched and the prefill launch takes every
  // request (so one with fewer queries, possible only when max_q
  // understates a request, is still computed).
  const int64_t min_q =
      static_cast<int64_t>(total_q) - static_cast<int64_t>(batch - 1) * max_q;
  pl.decode = min_q * G <= kDecodeRows;
  pl.prefill = static_cast<int64_t>(max_q) * G > kDecodeRows;
  if (!pl.decode) {
    pl.prefill_tiles = static_cast<int>(
        (static_cast<int64_t>(max_q) * G + 63) / 64);
    return pl;
  }
  if (pl.prefill)
    pl.prefill_tiles = static_cast<int>(
        (static_cast<int64_t>(max_q) * G + 63) / 64);
  // Widest key range a decode-class CTA can see.
  int64_t range = max_k;
  const int q_dec = kDecodeRows / G > 0 ? kDecodeRows / G : 1;
  if (wl >= 0) {
    const int64_t span = static_cast<int64_t>(wl) + q_dec +
                         (wr >= 0 ? wr : (causal ? 0 : max_k));
    if (span < range) range = span;
  }
  pl.range = range;
  // splits start on 64-key boundaries counted from the first admissible
  // key rounded down; with a left window that adds up to 63 keys of range
  const int64_t pad = wl >= 0 ? 63 : 0;
  if (fixed_split > 0) {
    // batch-invariant: fixed key ranges, always through the combine
    int64_t chunk = (static_cast<int64_t>(fixed_split) + kDecodeKT - 1) /
                    kDecodeKT * kDecodeKT;
    if (chunk > (1 << 30)) chunk = 1 << 30;
    pl.chunk = static_cast<int>(chunk);
    const int64_t n = range > 0 ? (range + pad + chunk - 1) / chunk : 1;
    pl.splits = static_cast<int>(n > 65535 ? 65535 : n);
  }
  int splits = 1;
  if (fixed_split > 0) {
    // plan made above
  } else if (num_splits > 1) {
    splits = num_splits;
  } else if (num_splits == 0 && range > 0) {
    // Split only to fill the GPU: with at least one (request, KV head) per
    // resident CTA slot the requests' own length spread balances the SMs,
    // and a split would only add partials and a combine.  Below that, cut
    // each range into as many pieces as keep every CTA resident in one
    // wave.  Keep >= 256 keys per split.
    const int64_t units = static_cast<int64_t>(batch) * Hkv;
    const int64_t slots = static_cast<int64_t>(sms) * kDecodeCtasPerSm;
    int64_t s = units >= slots ? 1 : slots / units;
    const int64_t cap = (range + 255) / 256;
    if (s > cap) s = cap;
    if (s > 64) s = 64;
    if (s < 1) s = 1;
    splits = static_cast<int>(s);
  }
  if (fixed_split <= 0 && splits > 1 && range > 0) {
    int64_t chunk = (range + splits - 1) / splits;
    chunk = (chunk + kDecodeKT - 1) / kDecodeKT * kDecodeKT;
    pl.chunk = static_cast<int>(chunk);
    pl.splits = static_cast<int>((range + pad + chunk - 1) / chunk);
    if (pl.splits <= 1) {
      pl.splits = 1;
      pl.chunk = 0;
    }
  }
  if (pl.chunk > 0) {
    // only decode-class requests (at most kDecodeRows / G tokens each)
    // write partials: rows per request when that is fewer than total_q
    const int tpr = kDecodeRows / G > 0 ? kDecodeRows / G : 1;
    const int64_t compact = static_cast<int64_t>(batch) * tpr;
    pl.part_tpr = compact < total_q ? tpr : 0;
    pl.part_rows = compact < total_q ? static_cast<int>(compact) : total_q;
    pl.part_o_bytes = align256(static_cast<size_t>(pl.splits) * pl.part_rows *
                               Hq * D * sizeof(float));
    pl.part_lse_bytes = align256(static_cast<size_t>(pl.splits) * Hq *
                                 pl.part_rows * sizeof(float));
    pl.workspace = pl.part_o_bytes + pl.part_lse_bytes;
  }
  return pl;
}

// Past the required workspace, calls with prefill-class requests take 256
// bytes more for the persistent prefill kernel's item counter, then, when
// the call has fewer prefill work items than SMs, room for that kernel's
// split-KV partials.  Both are optional: a workspace without them still
// runs, with a fixed item order and no split.
constexpr size_t kSchedBytes = 256;

// Key splits for the persistent prefill kernel (head size <= 128): only
// when even an upper bound of its work items, (ceil(total_q * G / 256) +
// batch) * Hkv, leaves half the SMs idle; as many as keep one wave, with
// at least 4 key tiles of 128 per split, at most 16.  Never with
// num_splits = 1 (no split asked for) or a fixed split size: the split
// depends on the rest of the batch, and those modes promise each request
// the same bits in any batch.
int prefill_splits(int batch, int total_q, int G, int Hkv, int max_k, int D,
                   int sms, int num_splits, int fixed_split) {
  if (D > 128 || num_splits == 1 || fixed_split > 0) return 1;
  const int64_t items =
      ((static_cast<int64_t>(total_q) * G + 255) / 256 + batch) * Hkv;
  if (items <= 0 || items * 2 > sms) return 1;
  int64_t s = sms / items;
  if (s > max_k / 512) s = max_k / 512;
  if (s > 16) s = 16;
  return s >= 2 ? static_cast<int>(s) : 1;
}
size_t prefill_split_bytes(int splits, int total_q, int Hq, int D) {
  if (splits <= 1) return 0;
  return align256(static_cast<size_t>(splits) * total_q * Hq * D * 4) +
         align256(static_cast<size_t>(splits) * Hq * total_q * 4);
}
// Calls that leave the split to the library (num_splits = 0, no fixed
// split size) run their decode-class requests on the persistent decode
// kernel when the workspace holds its scratch (the pieces of units that its
// CTA ranges cut); the scratch is sized for the larger of the 16-bit
// kernels' grids.
bool sk_candidate(int num_splits, int fixed_split, int D, bool kv8) {
  return num_splits == 0 && fixed_split <= 0 && decode_sk_supported(D, kv8);
}
int sk_rows(int G, int max_q) {
  const int64_t r = static_cast<int64_t>(G) * max_q;
  return r < kDecodeRows ? static_cast<int>(r) : kDecodeRows;
}
size_t sk_scratch_bytes(int D, bool kv8, bool q8, int sms, int rows) {
  int a = 0, b = 0;
  if (decode_sk_ctas(D, true, kv8, q8, sms, &a) != cudaSuccess ||
      decode_sk_ctas(D, false, kv8, q8, sms, &b) != cudaSuccess)
    return 0;
  return decode_sk_workspace_bytes(D, a > b ? a : b, rows);
}

// Workspace layout: the required part (decode split partials, fp8 page
// copies), then the optional tail: the persistent decode kernel's scratch
// (when the call may use it), and for calls with prefill-class requests
// the 256-byte item counter and the prefill split partials, last.
struct Layout {
  size_t need = 0;                    // required bytes
  size_t sk_off = 0, sk_bytes = 0;    // persistent decode scratch
  size_t sched_off = 0;               // prefill item counter (prefill only)
  size_t presplit_off = 0, presplit_bytes = 0;
  size_t total = 0;
};
Layout make_layout(size_t need, bool prefill, size_t sk_bytes,
                   size_t split_bytes) {
  Layout l;
  l.need = need;
  l.sk_off = align256(need);
  l.sk_bytes = sk_bytes;
  if (prefill) {
    l.sched_off = l.sk_off + sk_bytes;
    l.presplit_off = l.sched_off + kSchedBytes;
    l.presplit_bytes = split_bytes;
    l.total = l.presplit_off + split_bytes;
  } else {
    l.total = sk_bytes ? l.sk_off + sk_bytes : need;
  }
  return l;
}

// fp8 cache with prefill-class requests: 16-bit copies of up to
// batch * max_blocks pages (K and V) plus their block table.
size_t fp8_mock_bytes(int batch, int max_blocks, int BS, int Hkv, int D) {
  const size_t pages = static_cast<size_t>(batch) * max_blocks;
  return 2 * align256(pages * BS * Hkv * D * 2) + align256(pages * 4);
}
// fp8 query: a 16-bit copy of the codes [total_q, Hq, D], then 256 bytes
// holding k_scale * q_scale.
size_t q16_bytes(int total_q, int Hq, int D) {
  return align256(static_cast<size_t>(total_q) * Hq * D * 2) + 256;
}
bool q_fp8_of(const pkv_attention_options* o) { return o && o->q_fp8; }

bool non_paged(const pkv_attention_options* o) {
  return o && o->cu_seqlens_k;
}
int fixed_split_of(const pkv_attention_options* o) {
  return o ? o->fixed_split_size : 0;
}

pkv_status check_attn_shape(int batch, int total_q, int max_q, int max_k,
                            int Hq, int Hkv, int D, int BS, int num_splits) {
  if (batch < 0 || total_q < 0 || max_q < 0 || max_k < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size argument");
  if (Hq <= 0 || Hkv <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_heads and num_kv_heads must be > 0");
  if (Hq % Hkv != 0)
    return fail(PKV_ERR_INVALID_ARG,
                "num_heads (%d) must be a multiple of num_kv_heads (%d)", Hq,
                Hkv);
  if (BS <= 0 || BS % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "block_size must be a multiple of 16");
  if (D % 8 != 0 || D <= 0 || D > 256)
    return fail(PKV_ERR_UNSUPPORTED,
                "head_size %d: must be a multiple of 8 and at most 256", D);
  if (D != 64 && D != 128 && D != 256)
    return fail(PKV_ERR_UNSUPPORTED, "head_size %d not built (64, 128, 256)",
                D);
  if (num_splits < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_splits must be >= 0");
  return PKV_OK;
}

}  // namespace

// The workspace a call cannot do without (no prefill counter or split
// partials); the allocation-free entry point checks its scratch against it.
size_t required_workspace_bytes(int batch, int total_q, int max_seqlen_q,
                                int max_seqlen_k, int num_heads,
                                int num_kv_heads, int head_size,
                                int block_size, int causal, int window_left,
                                int window_right, int num_splits) {
  if (check_attn_shape(batch, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                       num_kv_heads, head_size, block_size,
                       num_splits) != PKV_OK)
    return static_cast<size_t>(-1);
  int sms = 0;
  if (device_info(nullptr, &sms) != PKV_OK) return static_cast<size_t>(-1);
  return make_plan(batch, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                   num_kv_heads, head_size, causal, window_left, window_right,
                   num_splits, sms)
      .workspace;
}

void set_last_error(const char* msg) { g_last_error = msg; }

cudaError_t smem_opt_in(const void* kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  constexpr int kSlots = 64;
  static const void* kerns[kSlots] = {};
  static uint64_t devs[kSlots] = {};      // bit d: done on device d
  std::lock_guard<std::mutex> lk(mu);
  int i = 0;
  while (i < kSlots && kerns[i] && kerns[i] != kern) ++i;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (i < kSlots && kerns[i] == kern && bit && (devs[i] & bit))
    return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e != cudaSuccess) return e;
  if (i < kSlots) {
    kerns[i] = kern;
    devs[i] |= bit;
  }
  return cudaSuccess;
}

int current_sm_count() {
  int sms = 0;
  if (device_info(nullptr, &sms) != PKV_OK || sms <= 0) return 1;
  return sms;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return g_last_error.c_str(); }

pkv_status pkv_set_prefill_kernel(int which) {
  if (which != PKV_PREFILL_TCGEN05 && which != PKV_PREFILL_MMA_SYNC &&
      which != PKV_PREFILL_TCGEN05_SMEM_P)
    return fail(PKV_ERR_INVALID_ARG, "unknown prefill kernel %d", which);
  g_prefill_kernel.store(which);
  return PKV_OK;
}

pkv_status pkv_set_decode_kernel(int which) {
  if (which != PKV_DECODE_TMA && which != PKV_DECODE_CP_ASYNC &&
      which != PKV_DECODE_PERSISTENT && which != PKV_DECODE_AUTO)
    return fail(PKV_ERR_INVALID_ARG, "unknown decode kernel %d", which);
  g_decode_kernel.store(which);
  return PKV_OK;
}

pkv_status pkv_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return PKV_OK;
}

uint64_t pkv_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}

pkv_status pkv_check_device_errors(pkv_stream_t stream) {
  unsigned* err = nullptr;
  pkv_status st = device_info(&err, nullptr);
  if (st != PKV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned host = 0;
  e = cudaMemcpy(&host, err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  const unsigned zero = 0;
  e = cudaMemcpy(err, &zero, sizeof(unsigned), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  if (!host) return PKV_OK;
  const char* what[] = {
      (host & kErrTimeout) ? " a bounded wait for data ran out (the CTA "
                             "drained its copies and stopped; its outputs "
                             "are not written);"
                           : "",
      (host & kErrBadBlock) ? " block id outside the cache (skipped);" : "",
      (host & kErrBadSlot) ? " slot outside the cache (skipped);" : "",
      (host & kErrBadTable)
          ? " key range beyond the table row or the K/V rows (clipped);"
          : "",
      (host & kErrQueryLen) ? " a request with more queries than "
                              "max_seqlen_q (not computed);"
                            : "",
      (host & kErrSmemAlign) ? " shared memory not 1024-byte aligned (the "
                               "kernel did nothing);"
                             : ""};
  const pkv_status code =
      (host & kErrTimeout)
          ? PKV_ERR_TIMEOUT
          : (host & (kErrBadBlock | kErrBadSlot | kErrBadTable | kErrQueryLen))
                ? PKV_ERR_BAD_INDEX
                : PKV_ERR_CUDA;
  return fail(code, "device error word 0x%x:%s%s%s%s%s%s", host, what[0],
              what[1], what[2], what[3], what[4], what[5]);
}

pkv_status pkv_reshape_and_cache(
    const void* key, const void* value, int64_t k_stride_tok,
    int64_t k_stride_head, int64_t v_stride_tok, int64_t v_stride_head,
    void* key_cache, void* value_cache, const int64_t cache_strides[4],
    const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
    int head_size, int block_size, int64_t num_blocks, pkv_dtype dtype,
    const char* kv_cache_dtype, const float* k_scale, const float* v_scale,
    pkv_stream_t stream) {
  bool fp8 = false;
  if (kv_cache_dtype && strcmp(kv_cache_dtype, "auto") != 0) {
    if (strcmp(kv_cache_dtype, "fp8") == 0 ||
        strcmp(kv_cache_dtype, "fp8_e4m3") == 0)
      fp8 = true;
    else
      return fail(PKV_ERR_UNSUPPORTED, "kv_cache_dtype '%s' is not supported",
                  kv_cache_dtype);
  }
  if (fp8 && (!k_scale || !v_scale))
    return fail(PKV_ERR_INVALID_ARG, "fp8 cache needs k_scale and v_scale");
  if (dtype != PKV_F16 && dtype != PKV_BF16)
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be fp16 or bf16");
  if (num_tokens < 0 || num_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size argument");
  if (num_kv_heads <= 0 || head_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_kv_heads / head_size must be > 0");
  if (block_size <= 0 || block_size % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "block_size must be a multiple of 16");
  if (head_size % 8 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "head_size must be a multiple of 8");
  if (!cache_strides)
    return fail(PKV_ERR_INVALID_ARG, "cache_strides is NULL");
  if (cache_strides[3] != 1)
    return fail(PKV_ERR_INVALID_ARG, "the head_size dim must be contiguous");
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  unsigned* err = nullptr;
  pkv_status st = device_info(&err, nullptr);
  if (st != PKV_OK) return st;
  cudaError_t e;
  if (fp8) {
    auto a16 = [](const void* ptr, int64_t st, int64_t sh, int eb) {
      return reinterpret_cast<uintptr_t>(ptr) % 16 == 0 &&
             (st * eb) % 16 == 0 && (sh * eb) % 16 == 0;
    };
    if (!a16(key, k_stride_tok, k_stride_head, 2) ||
        !a16(value, v_stride_tok, v_stride_head, 2) ||
        reinterpret_cast<uintptr_t>(key_cache) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(value_cache) % 8 != 0 ||
        cache_strides[0] % 8 || cache_strides[1] % 8 || cache_strides[2] % 8)
      return fail(PKV_ERR_UNSUPPORTED,
                  "fp8 cache write needs 16-byte aligned key/value rows and "
                  "8-byte aligned cache rows");
    e = launch_cache_write_fp8(
        key, value, k_stride_tok, k_stride_head, v_stride_tok, v_stride_head,
        key_cache, value_cache, cache_strides, slot_mapping, num_tokens,
        num_kv_heads, head_size, block_size, num_blocks, dtype == PKV_BF16,
        k_scale, v_scale, err, reinterpret_cast<cudaStream_t>(stream));
  } else {
    e = launch_cache_write(
        key, value, k_stride_tok, k_stride_head, v_stride_tok, v_stride_head,
        key_cache, value_cache, cache_strides, slot_mapping, num_tokens,
        num_kv_heads, head_size, block_size, num_blocks, 2, err,
        reinterpret_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  return PKV_OK;
}

}  // extern "C"

namespace {

// Workspace of an attention call; pre_splits > 0 fixes the prefill key
// splits (else the plan's).
size_t workspace_bytes_impl(int batch, int total_q, int max_seqlen_q,
                            int max_seqlen_k, int num_heads, int num_kv_heads,
                            int head_size, int block_size, int causal,
                            int window_left, int window_right, int num_splits,
                            int max_blocks_per_seq,
                            const pkv_attention_options* opts,
                            int pre_splits) {
  const int bs = non_paged(opts) ? 16 : block_size;
  if (check_attn_shape(batch, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                       num_kv_heads, head_size, bs, num_splits) != PKV_OK)
    return static_cast<size_t>(-1);
  if (fixed_split_of(opts) < 0 || (fixed_split_of(opts) > 0 && num_splits))
    return static_cast<size_t>(-1);
  int sms = 0;
  if (device_info(nullptr, &sms) != PKV_OK) return static_cast<size_t>(-1);
  const Plan pl =
      make_plan(batch, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                num_kv_heads, head_size, causal,
                window_left < 0 ? -1 : window_left,
                window_right < 0 ? -1 : window_right, num_splits, sms,
                fixed_split_of(opts));
  const bool fp8 = opts && opts->kv_cache_fp8;
  const size_t split_bytes = prefill_split_bytes(
      !pl.prefill ? 1
      : pre_splits > 0
          ? pre_splits
          : prefill_splits(batch, total_q, num_heads / num_kv_heads,
                           num_kv_heads, max_seqlen_k, head_size, sms,
                           num_splits, fixed_split_of(opts)),
      total_q, num_heads, head_size);
  const bool q8 = fp8 && q_fp8_of(opts);
  const size_t skb =
      sk_candidate(num_splits, fixed_split_of(opts), head_size, fp8)
          ? sk_scratch_bytes(head_size, fp8, q8, sms,
                             sk_rows(num_heads / num_kv_heads, max_seqlen_q))
          : 0;
  size_t need = pl.workspace;
  if (fp8 && pl.prefill) {
    if (max_blocks_per_seq <= 0) return static_cast<size_t>(-1);
    need = align256(pl.workspace) +
           fp8_mock_bytes(batch, max_blocks_per_seq, block_size, num_kv_heads,
                          head_size);
  }
  if (q8) need = align256(need) + q16_bytes(total_q, num_heads, head_size);
  return make_layout(need, pl.prefill, skb, split_bytes).total;
}

}  // namespace

extern "C" {

size_t pkv_paged_attention_workspace_size_opts(
    int batch, int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
    int num_kv_heads, int head_size, int block_size, int causal,
    int window_left, int window_right, int num_splits,
    int max_blocks_per_seq, const pkv_attention_options* opts) {
  return workspace_bytes_impl(batch, total_q, max_seqlen_q, max_seqlen_k,
                              num_heads, num_kv_heads, head_size, block_size,
                              causal, window_left, window_right, num_splits,
                              max_blocks_per_seq, opts, 0);
}

size_t pkv_paged_attention_workspace_size(int batch, int total_q,
                                          int max_seqlen_q, int max_seqlen_k,
                                          int num_heads, int num_kv_heads,
                                          int head_size, int block_size,
                                          int causal, int window_left,
                                          int window_right, int num_splits) {
  if (check_attn_shape(batch, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                       num_kv_heads, head_size, block_size,
                       num_splits) != PKV_OK)
    return static_cast<size_t>(-1);
  int sms = 0;
  if (device_info(nullptr, &sms) != PKV_OK) return static_cast<size_t>(-1);
  const Plan pl = make_plan(batch, total_q, max_seqlen_q, max_seqlen_k,
                            num_heads, num_kv_heads, head_size, causal,
                            window_left, window_right, num_splits, sms);
  const size_t split_bytes = prefill_split_bytes(
      pl.prefill ? prefill_splits(batch, total_q, num_heads / num_kv_heads,
                                  num_kv_heads, max_seqlen_k, head_size, sms,
                                  num_splits, 0)
                 : 1,
      total_q, num_heads, head_size);
  const size_t skb =
      sk_candidate(num_splits, 0, head_size, false)
          ? sk_scratch_bytes(head_size, false, false, sms,
                             sk_rows(num_heads / num_kv_heads, max_seqlen_q))
          : 0;
  return make_layout(pl.workspace, pl.prefill, skb, split_bytes).total;
}

pkv_status pkv_paged_attention_varlen(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], void* out, int64_t o_stride_tok,
    int64_t o_stride_head, const int32_t* cu_seqlens_q,
    const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q,
    int max_seqlen_k, const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, float softmax_scale, int causal,
    int window_left, int window_right, float softcap,
    const float* alibi_slopes, int num_splits, float* softmax_lse,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype,
    pkv_stream_t stream) {
  return pkv_paged_attention_varlen_opts(
      q, q_stride_tok, q_stride_head, key_cache, value_cache, cache_strides,
      out, o_stride_tok, o_stride_head, cu_seqlens_q, seqused_k, batch,
      total_q, max_seqlen_q, max_seqlen_k, block_table, block_table_stride,
      max_blocks_per_seq, num_heads, num_kv_heads, head_size, block_size,
      num_blocks, softmax_scale, causal, window_left, window_right, softcap,
      alibi_slopes, num_splits, softmax_lse, workspace, workspace_bytes,
      dtype, stream, nullptr);
}

}  // extern "C"

namespace {

// Controls of an attention call inside a composed one (the cascade).
struct Internal {
  // launch the TMA decode kernel (when the call takes it) as a programmatic
  // dependent of the grid queued before the call, with this zeroed counter
  int* pdl_done = nullptr;
  int pre_splits = 0;       // > 0: prefill key splits (else the plan's)
  int pre_ctas = 0;         // > 0: cap on the persistent prefill grid
  // leave the prefill split combine to the caller (filled in below)
  bool defer_combine = false;
  bool deferred = false;
  CombineParams combine{};
  int combine_max_q = 0;
  bool combine_bf16 = false;
  // set by the call: a workspace int it zeroed before its first kernel and
  // does not use itself (null if none)
  int* zeroed_counter = nullptr;
};

pkv_status attention_impl(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], void* out, int64_t o_stride_tok,
    int64_t o_stride_head, const int32_t* cu_seqlens_q,
    const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q,
    int max_seqlen_k, const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, float softmax_scale, int causal,
    int window_left, int window_right, float softcap,
    const float* alibi_slopes, int num_splits, float* softmax_lse,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype,
    pkv_stream_t stream, const pkv_attention_options* opts, Internal* in) {
  int* pdl_done = in ? in->pdl_done : nullptr;
  const bool nonpaged = non_paged(opts);
  pkv_status st = check_attn_shape(batch, total_q, max_seqlen_q, max_seqlen_k,
                                   num_heads, num_kv_heads, head_size,
                                   nonpaged ? 16 : block_size, num_splits);
  if (st != PKV_OK) return st;
  const int fixed_split = fixed_split_of(opts);
  if (fixed_split < 0)
    return fail(PKV_ERR_INVALID_ARG, "fixed_split_size must be >= 0");
  if (fixed_split > 0 && num_splits != 0)
    return fail(PKV_ERR_INVALID_ARG,
                "fixed_split_size and num_splits are exclusive");
  if (dtype != PKV_F16 && dtype != PKV_BF16)
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be fp16 or bf16");
  if (!(softmax_scale == softmax_scale) || isinf(softmax_scale))
    return fail(PKV_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (softcap < 0.f || !(softcap == softcap))
    return fail(PKV_ERR_INVALID_ARG, "softcap must be >= 0 (0 = none)");
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!q || !key_cache || !value_cache || !out || !cu_seqlens_q ||
      !cache_strides)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!nonpaged && (!seqused_k || !block_table))
    return fail(PKV_ERR_INVALID_ARG, "NULL seqused_k or block_table");
  if (!nonpaged &&
      (max_blocks_per_seq <= 0 || block_table_stride < max_blocks_per_seq))
    return fail(PKV_ERR_INVALID_ARG,
                "block_table: need max_blocks_per_seq >= 1 and stride >= it");
  if (cache_strides[3] != 1)
    return fail(PKV_ERR_INVALID_ARG, "the head_size dim must be contiguous");
  const bool kv8 = opts && opts->kv_cache_fp8;
  if (nonpaged && kv8)
    return fail(PKV_ERR_UNSUPPORTED,
                "an fp8 cache is not supported for non-paged attention");
  if (nonpaged && opts->total_k < 0)
    return fail(PKV_ERR_INVALID_ARG, "total_k must be >= 0");
  if (nonpaged && (cache_strides[1] <= 0 || cache_strides[2] <= 0))
    return fail(PKV_ERR_INVALID_ARG, "non-paged K/V strides must be > 0");
  if (kv8 && (!opts->k_scale || !opts->v_scale))
    return fail(PKV_ERR_INVALID_ARG, "fp8 cache needs k_scale and v_scale");
  if (kv8 && head_size % 16 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "fp8 cache needs head_size % 16 == 0");
  const bool q8 = q_fp8_of(opts);
  if (q8 && !kv8)
    return fail(PKV_ERR_UNSUPPORTED, "an fp8 query needs an fp8 cache");
  if (q8 && !opts->q_scale)
    return fail(PKV_ERR_INVALID_ARG, "an fp8 query needs q_scale");
  const int eb = 2, cb = kv8 ? 1 : 2, qb = q8 ? 1 : 2;
  if (!aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned16(out) || !stride16(q_stride_tok, qb) ||
      !stride16(q_stride_head, qb) || !stride16(o_stride_tok, eb) ||
      !stride16(o_stride_head, eb) ||
      !stride16(nonpaged ? 0 : cache_strides[0], cb) ||
      !stride16(cache_strides[1], cb) || !stride16(cache_strides[2], cb))
    return fail(PKV_ERR_UNSUPPORTED,
                "q/out/cache rows must start on 16-byte boundaries");
  const int wl = window_left < 0 ? -1 : window_left;
  const int wr = window_right < 0 ? -1 : window_right;

  unsigned* err = nullptr;
  int sms = 0;
  st = device_info(&err, &sms);
  if (st != PKV_OK) return st;
  const Plan pl = make_plan(batch, total_q, max_seqlen_q, max_seqlen_k,
                            num_heads, num_kv_heads, head_size, causal, wl, wr,
                            num_splits, sms, fixed_split);
  size_t need = pl.workspace;
  size_t mock_off = 0, q16_off = 0;
  if (kv8 && pl.prefill) {
    mock_off = align256(pl.workspace);
    need = mock_off + fp8_mock_bytes(batch, max_blocks_per_seq, block_size,
                                     num_kv_heads, head_size);
  }
  if (q8) {
    q16_off = align256(need);
    need = q16_off + q16_bytes(total_q, num_heads, head_size);
  }
  if (need > 0) {
    if (workspace_bytes < need || !workspace)
      return fail(PKV_ERR_WORKSPACE_TOO_SMALL,
                  "workspace of %zu bytes needed, %zu given", need,
                  workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
      return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  // optional tail: the persistent decode scratch, then the prefill item
  // counter and its split partials
  const int sp = !pl.prefill ? 1
                 : (in && in->pre_splits > 0)
                     ? in->pre_splits
                     : prefill_splits(batch, total_q, num_heads / num_kv_heads,
                                      num_kv_heads, max_seqlen_k, head_size,
                                      sms, num_splits, fixed_split);
  const size_t sb = prefill_split_bytes(sp, total_q, num_heads, head_size);
  // Persistent or one CTA per (request, KV head, split)?  Measured on
  // GB300: when the (request, KV head) units fill about one wave of the
  // per-unit kernel's resident CTAs, the hardware's dealing of CTAs to SMs
  // balances the SMs better than equal static shares (batched decode,
  // 512 units: 0.1131 against 0.1157 ms), and so it does for many short
  // units (cascade suffix, 2048 units of 512 keys: 0.2095 against 0.2181
  // ms for the whole cascade); from two waves of long units on the
  // persistent kernel is ahead (124 windowed D = 256 decodes, 992 units of
  // up to 4096 keys: 0.581 against 0.625 ms).  fp8 caches always take it
  // (the per-unit fp8 kernel is 1.9 times slower).
  const int dsel = g_decode_kernel.load();
  const bool many_units =
      static_cast<int64_t>(batch) * num_kv_heads >=
          2 * static_cast<int64_t>(sms) * kDecodeCtasPerSm &&
      pl.range >= kLongUnitKeys;
  const bool sk_ok =
      sk_candidate(num_splits, fixed_split, head_size, kv8) &&
      (dsel == PKV_DECODE_PERSISTENT ||
       (dsel == PKV_DECODE_AUTO && (kv8 || many_units)));
  const int skr = sk_rows(num_heads / num_kv_heads, max_seqlen_q);
  const size_t skb = sk_candidate(num_splits, fixed_split, head_size, kv8)
                         ? sk_scratch_bytes(head_size, kv8, q8, sms, skr)
                         : 0;
  const Layout lay = make_layout(need, pl.prefill, skb, sb);
  const bool ws_ok = workspace &&
                     reinterpret_cast<uintptr_t>(workspace) % 256 == 0;
  int sk_ctas = 0;
  void* sk_scratch = nullptr;
  if (sk_ok && pl.decode && skb > 0 && ws_ok &&
      workspace_bytes >= lay.sk_off + lay.sk_bytes) {
    if (decode_sk_ctas(head_size, dtype == PKV_BF16, kv8, q8, sms,
                       &sk_ctas) ==
            cudaSuccess &&
        decode_sk_workspace_bytes(head_size, sk_ctas, skr) <= lay.sk_bytes)
      sk_scratch = static_cast<char*>(workspace) + lay.sk_off;
    else
      sk_ctas = 0;
  }
  int* sched = nullptr;
  int pre_splits = 1;
  float* pre_o = nullptr;
  float* pre_lse = nullptr;
  if (pl.prefill && ws_ok) {
    char* wsc = static_cast<char*>(workspace);
    if (workspace_bytes >= lay.sched_off + kSchedBytes)
      sched = reinterpret_cast<int*>(wsc + lay.sched_off);
    if (sp > 1 && workspace_bytes >= lay.presplit_off + lay.presplit_bytes) {
      pre_splits = sp;
      pre_o = reinterpret_cast<float*>(wsc + lay.presplit_off);
      pre_lse = reinterpret_cast<float*>(
          wsc + lay.presplit_off +
          align256(static_cast<size_t>(sp) * total_q * num_heads *
                   head_size * 4));
    }
  }

  AttnParams p{};
  p.q = q;
  p.q_st = q_stride_tok;
  p.q_sh = q_stride_head;
  p.kc = key_cache;
  p.vc = value_cache;
  p.c_sb = cache_strides[0];
  p.c_sr = cache_strides[1];
  p.c_sh = cache_strides[2];
  p.out = out;
  p.o_st = o_stride_tok;
  p.o_sh = o_stride_head;
  p.lse = softmax_lse;
  p.total_q = total_q;
  p.cu_q = cu_seqlens_q;
  p.seqused_k = seqused_k;
  p.batch = batch;
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.Hq = num_heads;
  p.Hkv = num_kv_heads;
  p.G = num_heads / num_kv_heads;
  p.BS = block_size;
  p.bs_shift = -1;
  if ((block_size & (block_size - 1)) == 0)
    for (int sh = 0; sh < 31; ++sh)
      if ((1 << sh) == block_size) p.bs_shift = sh;
  p.scale = softmax_scale;
  p.softcap = softcap;
  p.alibi = alibi_slopes;
  p.sinks = opts ? opts->sinks : nullptr;
  p.kv_fp8 = kv8 ? 1 : 0;
  p.k_scale = kv8 ? opts->k_scale : nullptr;
  p.v_scale = kv8 ? opts->v_scale : nullptr;
  if (nonpaged) {
    // one "block" holding all total_k rows; kernels index rows by cu_k
    const int rows = opts->total_k > 0 ? opts->total_k : 1;
    p.cu_k = opts->cu_seqlens_k;
    p.total_k = opts->total_k;
    p.block_table = nullptr;
    p.bt_stride = 0;
    p.max_blocks = 1;
    p.num_blocks = 1;
    p.BS = rows;
    p.bs_shift = -1;
    const int64_t ext_r = static_cast<int64_t>(rows) * p.c_sr;
    const int64_t ext_h = static_cast<int64_t>(num_kv_heads) * p.c_sh;
    p.c_sb = ext_r > ext_h ? ext_r : ext_h;
  }
  p.causal = causal ? 1 : 0;
  p.wl = wl;
  p.wr = wr;
  p.err = err;
  p.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  const bool bf16 = dtype == PKV_BF16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // fp8 query: the persistent decode kernel reads the codes; every other
  // kernel reads their exact 16-bit copy, with k_scale * q_scale as k_scale
  AttnParams p16 = p;
  if (q8 && (pl.prefill || sk_scratch == nullptr)) {
    char* base_ptr = static_cast<char*>(workspace) + q16_off;
    float* kq = reinterpret_cast<float*>(
        base_ptr + align256(static_cast<size_t>(total_q) * num_heads *
                            head_size * 2));
    cudaError_t e = launch_widen_q(q, q_stride_tok, q_stride_head, base_ptr,
                                   total_q, num_heads, head_size,
                                   opts->k_scale, opts->q_scale, kq, bf16, s);
    if (e != cudaSuccess) return cuda_fail(e, "fp8 query copy launch");
    p16.q = base_ptr;
    p16.q_st = static_cast<int64_t>(num_heads) * head_size;
    p16.q_sh = head_size;
    p16.k_scale = kq;
  }
  if (q8) {
    p.q_fp8 = 1;
    p.q_scale = opts->q_scale;
  }

  const int which = g_prefill_kernel.load();
  const bool tc_prefill =
      which == PKV_PREFILL_TCGEN05 || which == PKV_PREFILL_TCGEN05_SMEM_P;
  // Prefill first: the persistent prefill kernel takes every SM, and the
  // decode-class requests' kernel (the one-CTA-per-unit TMA decode kernel)
  // is its programmatic dependent, so that its CTAs run in the prefill's
  // tail.  The decode grid's last CTA waits for the prefill grid (a counter
  // beside the item counter), so whatever follows in the stream still sees
  // both done.  The two write disjoint rows of the output.
  // no_pdl: every kernel of the call in plain stream order
  const bool pdl_ok = !(opts && opts->no_pdl);
  const bool prefill_first = pdl_ok && pl.prefill && pl.decode && sched &&
                             tc_prefill && sk_scratch == nullptr && !kv8 &&
                             dsel != PKV_DECODE_CP_ASYNC &&
                             pdl_done == nullptr;
  // the prefill kernel's item counter (and the counter above) is zeroed
  // before any decode kernel, so that the prefill launch can follow those
  // kernels directly
  bool sched_zeroed = false;
  if (pl.prefill && sched) {
    cudaError_t e = cudaMemsetAsync(sched, 0, 2 * sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    sched_zeroed = true;
    // the second counter is free for the caller unless this call uses it
    if (in && !prefill_first) in->zeroed_counter = sched + 1;
  }

  // the decode-class requests; done: the counter of the decode grid's CTAs
  // when it is a programmatic dependent of the launch before it
  auto run_decode = [&](int* done) -> pkv_status {
    AttnParams d = sk_scratch ? p : p16;
    d.min_rows = 1;
    d.max_rows = kDecodeRows;
    d.chunk = pl.chunk;
    d.part_tpr = pl.part_tpr;
    d.part_rows = pl.part_rows;
    if (pl.chunk > 0) {
      d.part_o = static_cast<float*>(workspace);
      d.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                            pl.part_o_bytes);
    }
    cudaError_t e;
    const bool persistent = sk_scratch != nullptr;
    if (persistent) {
      d.chunk = 0;
      e = launch_decode_attn_sk(d, head_size, bf16, sk_ctas, skr, sk_scratch,
                                pdl_ok, s);
    } else if ((!kv8 || head_size == 128) && dsel != PKV_DECODE_CP_ASYNC) {
      d.pdl_done = done;
      e = launch_decode_attn_tma(d, head_size, bf16, pl.splits, s);
    } else {
      e = launch_decode_attn(d, head_size, bf16, pl.splits, 1, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    if (pl.chunk > 0 && !persistent) {
      CombineParams c{};
      c.part_o = d.part_o;
      c.part_lse = d.part_lse;
      c.part_tpr = pl.part_tpr;
      c.part_rows = pl.part_rows;
      c.out = out;
      c.o_st = o_stride_tok;
      c.o_sh = o_stride_head;
      c.lse = softmax_lse;
      c.total_q = total_q;
      c.cu_q = cu_seqlens_q;
      c.seqused_k = seqused_k;
      c.cu_k = p.cu_k;
      c.batch = batch;
      c.Hq = num_heads;
      c.G = p.G;
      c.D = head_size;
      c.causal = p.causal;
      c.wl = wl;
      c.wr = wr;
      c.chunk = pl.chunk;
      c.splits = pl.splits;
      c.sinks = p.sinks;
      c.min_rows = 1;
      c.max_rows = kDecodeRows;
      // a dependent of the decode grid when that is one itself
      e = launch_split_combine(c, bf16, s, done != nullptr);
      if (e != cudaSuccess) return cuda_fail(e, "split combine launch");
    }
    return PKV_OK;
  };

  auto run_prefill = [&]() -> pkv_status {
    AttnParams f = p16;
    f.min_rows = pl.decode ? kDecodeRows + 1 : 1;
    f.max_rows = 0x7fffffff;
    f.chunk = 0;
    f.sched = sched;
    f.sched_zeroed = sched_zeroed ? 1 : 0;
    f.pre_splits = pre_splits;
    f.pre_o = pre_o;
    f.pre_lse = pre_lse;
    f.max_ctas = in ? in->pre_ctas : 0;
    const int64_t prow = static_cast<int64_t>(max_seqlen_q) * p.G;
    cudaError_t e;
    if (kv8) {
      // 16-bit copies of the pages prefill-class requests read
      const size_t pages = static_cast<size_t>(batch) * max_blocks_per_seq;
      const size_t page_bytes =
          static_cast<size_t>(block_size) * num_kv_heads * head_size * 2;
      char* base_ptr = static_cast<char*>(workspace) + mock_off;
      void* mk = base_ptr;
      void* mv = base_ptr + align256(pages * page_bytes);
      int32_t* mt = reinterpret_cast<int32_t*>(
          base_ptr + 2 * align256(pages * page_bytes));
      e = launch_fp8_dequant_pages(f, head_size, bf16, mk, mv, mt, s);
      if (e != cudaSuccess) return cuda_fail(e, "fp8 page dequant launch");
      f.kc = mk;
      f.vc = mv;
      f.c_sb = static_cast<int64_t>(block_size) * num_kv_heads * head_size;
      f.c_sr = static_cast<int64_t>(num_kv_heads) * head_size;
      f.c_sh = head_size;
      f.block_table = mt;
      f.bt_stride = max_blocks_per_seq;
      f.num_blocks = static_cast<int64_t>(pages);
      f.kv_fp8 = 0;          // 16-bit copies; k_scale / v_scale still apply
    }
    int used = 1;
    if (tc_prefill)
      // as a programmatic dependent of the decode kernels just launched
      // (none of their output is read here); not after an fp8 page copy,
      // which this launch reads
      e = launch_prefill_attn_tc(f, head_size, bf16,
                                 static_cast<int>((prow + 127) / 128),
                                 which == PKV_PREFILL_TCGEN05, &used, s,
                                 pdl_ok && PKV_PREFILL_AFTER_DECODE_PDL &&
                                     pl.decode &&
                                     !kv8 && !prefill_first);
    else
      e = launch_prefill_attn_mma(f, head_size, bf16,
                                  static_cast<int>((prow + 63) / 64), s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
    if (used > 1) {
      CombineParams c{};
      c.part_o = pre_o;
      c.part_lse = pre_lse;
      c.part_tpr = 0;              // prefill partials: one row per token
      c.part_rows = total_q;
      c.out = out;
      c.o_st = o_stride_tok;
      c.o_sh = o_stride_head;
      c.lse = softmax_lse;
      c.total_q = total_q;
      c.cu_q = cu_seqlens_q;
      c.batch = batch;
      c.Hq = num_heads;
      c.G = p.G;
      c.D = head_size;
      c.splits = used;
      c.sinks = p.sinks;
      c.min_rows = f.min_rows;
      c.max_rows = 0x7fffffff;
      if (in && in->defer_combine) {
        in->deferred = true;
        in->combine = c;
        in->combine_max_q = max_seqlen_q;
        in->combine_bf16 = bf16;
      } else {
        e = launch_prefill_split_combine(c, max_seqlen_q, bf16, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill split combine");
      }
    }
    return PKV_OK;
  };

  pkv_status rc = PKV_OK;
  if (prefill_first) {
    rc = run_prefill();
    if (rc == PKV_OK) rc = run_decode(sched + 1);
  } else {
    if (pl.decode) rc = run_decode(pdl_done);
    if (rc == PKV_OK && pl.prefill) rc = run_prefill();
  }
  return rc;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_varlen_opts(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], void* out, int64_t o_stride_tok,
    int64_t o_stride_head, const int32_t* cu_seqlens_q,
    const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q,
    int max_seqlen_k, const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, float softmax_scale, int causal,
    int window_left, int window_right, float softcap,
    const float* alibi_slopes, int num_splits, float* softmax_lse,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype,
    pkv_stream_t stream, const pkv_attention_options* opts) {
  return attention_impl(
      q, q_stride_tok, q_stride_head, key_cache, value_cache, cache_strides,
      out, o_stride_tok, o_stride_head, cu_seqlens_q, seqused_k, batch,
      total_q, max_seqlen_q, max_seqlen_k, block_table, block_table_stride,
      max_blocks_per_seq, num_heads, num_kv_heads, head_size, block_size,
      num_blocks, softmax_scale, causal, window_left, window_right, softcap,
      alibi_slopes, num_splits, softmax_lse, workspace, workspace_bytes,
      dtype, stream, opts, nullptr);
}

pkv_status pkv_scaled_fp8_quant(const void* in, int64_t in_row_stride,
                                void* out, int64_t out_row_stride,
                                int64_t rows, int cols, const float* scale,
                                pkv_dtype dtype, pkv_stream_t stream) {
  if (dtype != PKV_F16 && dtype != PKV_BF16)
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be fp16 or bf16");
  if (rows < 0 || cols < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size argument");
  if (cols % 16 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "cols must be a multiple of 16");
  if (rows == 0 || cols == 0) return PKV_OK;
  if (!in || !out || !scale)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (in_row_stride < cols || out_row_stride < cols)
    return fail(PKV_ERR_INVALID_ARG, "row strides must be >= cols");
  if (!aligned16(in) || !aligned16(out) || !stride16(in_row_stride, 2) ||
      !stride16(out_row_stride, 1))
    return fail(PKV_ERR_UNSUPPORTED,
                "rows must start on 16-byte boundaries");
  cudaError_t e = launch_scaled_fp8_quant(
      in, in_row_stride, out, out_row_stride, rows, cols, scale,
      dtype == PKV_BF16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scaled_fp8_quant launch");
  return PKV_OK;
}

// Cascade prefix: key splits of the prefill kernel and the SMs its grid
// leaves to the suffix's decode kernel (0: the grid is not capped).
// Measured on GB300 (256 decodes over an 8192-key prefix + 512 own keys,
// 64/8 heads): unsplit and uncapped 0.134 ms (the prefix's 64 items take
// 64 SMs and the suffix the other 88); 2 splits leaving 24 or 56 SMs 0.170
// and 0.162 ms; 3 splits leaving 40 or 56 SMs 0.162 and 0.161 ms; 4 splits
// leaving 24 or 56 SMs 0.178 and 0.166 ms.
#ifndef PKV_CASCADE_PREFIX_SPLITS
#define PKV_CASCADE_PREFIX_SPLITS 1
#endif
#ifndef PKV_CASCADE_SUFFIX_SMS
#define PKV_CASCADE_SUFFIX_SMS 0
#endif

// Cascade: the workspace holds, in order, a 256-byte counter block, the
// prefix and suffix outputs (16-bit [T, Hq, D]) and LSEs (fp32 [Hq, T]),
// then the prefix call's workspace and the suffix call's.
struct CascadeLayout {
  size_t po = 0, pl = 0, so = 0, sl = 0, pws = 0, sws = 0, total = 0;
  size_t pws_bytes = 0, sws_bytes = 0;
};

static bool cascade_layout(int batch, int T, int max_q, int max_kv, int P,
                           int Hq, int Hkv, int D, int BS, int max_blocks,
                           int num_splits, const pkv_attention_options* o,
                           CascadeLayout* l) {
  const size_t out_b = align256(static_cast<size_t>(T) * Hq * D * 2);
  const size_t lse_b = align256(static_cast<size_t>(Hq) * T * 4);
  l->po = 256;
  l->pl = l->po + out_b;
  l->so = l->pl + lse_b;
  l->sl = l->so + out_b;
  l->pws = l->sl + lse_b;
  const int nc = BS > 0 ? P / BS : 0;
  l->pws_bytes = workspace_bytes_impl(1, T, T, P, Hq, Hkv, D, BS, 0, -1, -1,
                                      1, nc, o, PKV_CASCADE_PREFIX_SPLITS);
  l->sws_bytes = pkv_paged_attention_workspace_size_opts(
      batch, T, max_q, max_kv - P, Hq, Hkv, D, BS, 1, -1, -1, num_splits,
      max_blocks - nc, o);
  if (l->pws_bytes == static_cast<size_t>(-1) ||
      l->sws_bytes == static_cast<size_t>(-1))
    return false;
  l->sws = l->pws + align256(l->pws_bytes);
  l->total = l->sws + align256(l->sws_bytes);
  return true;
}

size_t pkv_cascade_attention_workspace_size(
    int batch, int num_tokens, int max_query_len, int max_kv_len,
    int common_prefix_len, int num_heads, int num_kv_heads, int head_size,
    int block_size, int max_blocks_per_seq, int num_splits,
    const pkv_attention_options* opts) {
  if (block_size <= 0 || common_prefix_len <= 0 ||
      common_prefix_len % block_size != 0 || max_kv_len < common_prefix_len ||
      max_blocks_per_seq < common_prefix_len / block_size)
    return static_cast<size_t>(-1);
  CascadeLayout l;
  if (!cascade_layout(batch, num_tokens, max_query_len, max_kv_len,
                      common_prefix_len, num_heads, num_kv_heads, head_size,
                      block_size, max_blocks_per_seq, num_splits, opts, &l))
    return static_cast<size_t>(-1);
  return l.total;
}

pkv_status pkv_cascade_attention(
    void* output, const void* query, int64_t q_stride_tok,
    int64_t q_stride_head, const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], const int32_t* cu_query_lens,
    int max_query_len, const int32_t* cu_prefix_query_lens,
    const int32_t* prefix_kv_lens, const int32_t* suffix_kv_lens,
    int max_kv_len, int batch, int num_tokens, float softmax_scale,
    float logits_soft_cap, const int32_t* block_table,
    int64_t block_table_stride, int max_blocks_per_seq,
    int common_prefix_len, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, int num_splits, int overlap,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype,
    pkv_stream_t stream, const pkv_attention_options* opts) {
  if (opts && (opts->cu_seqlens_k || opts->fixed_split_size))
    return fail(PKV_ERR_INVALID_ARG,
                "cascade attention takes no cu_seqlens_k or fixed split");
  if (dtype != PKV_F16 && dtype != PKV_BF16)
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be fp16 or bf16");
  if (block_size <= 0 || common_prefix_len <= 0 ||
      common_prefix_len % block_size != 0)
    return fail(PKV_ERR_INVALID_ARG,
                "common_prefix_len must be a positive multiple of "
                "block_size");
  if (max_kv_len < common_prefix_len ||
      max_blocks_per_seq < common_prefix_len / block_size)
    return fail(PKV_ERR_INVALID_ARG,
                "the prefix is longer than max_kv_len or the table");
  if (batch < 0 || num_tokens < 0 || num_splits < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size argument");
  if (batch == 0 || num_tokens == 0) return PKV_OK;
  if (!output || !cu_prefix_query_lens || !prefix_kv_lens ||
      !suffix_kv_lens || !block_table)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  CascadeLayout l;
  if (!cascade_layout(batch, num_tokens, max_query_len, max_kv_len,
                      common_prefix_len, num_heads, num_kv_heads, head_size,
                      block_size, max_blocks_per_seq, num_splits, opts, &l))
    return fail(PKV_ERR_INVALID_ARG,
                "invalid shapes for the prefix or suffix attention");
  if (!workspace || workspace_bytes < l.total)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL,
                "workspace of %zu bytes needed, %zu given", l.total,
                workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!aligned16(output))
    return fail(PKV_ERR_UNSUPPORTED, "output must be 16-byte aligned");
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = num_tokens, Hq = num_heads, D = head_size;
  const int nc = common_prefix_len / block_size;
  void* po = ws + l.po;
  float* pl = reinterpret_cast<float*>(ws + l.pl);
  void* so = ws + l.so;
  float* sl = reinterpret_cast<float*>(ws + l.sl);
  // prefix: every query over the shared blocks (row 0 of the table),
  // non-causal, with the sinks; its grid leaves SMs to the suffix, and its
  // split combine (if any) waits until the suffix's decode is queued
  int sms = 0;
  pkv_status st = device_info(nullptr, &sms);
  if (st != PKV_OK) return st;
  Internal pin;
  pin.pre_splits = PKV_CASCADE_PREFIX_SPLITS;
  pin.pre_ctas = PKV_CASCADE_SUFFIX_SMS > 0 && sms > PKV_CASCADE_SUFFIX_SMS
                     ? sms - PKV_CASCADE_SUFFIX_SMS
                     : 0;
  pin.defer_combine = true;
  st = attention_impl(
      query, q_stride_tok, q_stride_head, key_cache, value_cache,
      cache_strides, po, static_cast<int64_t>(Hq) * D, D,
      cu_prefix_query_lens, prefix_kv_lens, 1, T, T, common_prefix_len,
      block_table, block_table_stride, nc, Hq, num_kv_heads, D, block_size,
      num_blocks, softmax_scale, 0, -1, -1, logits_soft_cap, nullptr, 1, pl,
      ws + l.pws, l.pws_bytes, dtype, stream, opts, &pin);
  if (st != PKV_OK) return st;
  // the suffix decode grid's CTA counter: one the prefix call zeroed before
  // its kernel, so that nothing comes between the prefix kernel and the
  // suffix decode kernel that depends on it; else one zeroed here (correct,
  // without the overlap)
  int* done = nullptr;
  if (overlap) {
    done = pin.zeroed_counter;
    if (!done) {
      done = reinterpret_cast<int*>(ws);
      cudaError_t e = cudaMemsetAsync(done, 0, sizeof(int), s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    }
  }
  // suffix: each request's own blocks, causal, without the sinks; its
  // decode kernel may start beside the prefix kernel
  pkv_attention_options so_opts{};
  if (opts) so_opts = *opts;
  so_opts.sinks = nullptr;
  Internal sin;
  sin.pdl_done = overlap ? done : nullptr;
  st = attention_impl(
      query, q_stride_tok, q_stride_head, key_cache, value_cache,
      cache_strides, so, static_cast<int64_t>(Hq) * D, D, cu_query_lens,
      suffix_kv_lens, batch, T, max_query_len, max_kv_len - common_prefix_len,
      block_table + nc, block_table_stride, max_blocks_per_seq - nc, Hq,
      num_kv_heads, D, block_size, num_blocks, softmax_scale, 1, -1, -1,
      logits_soft_cap, nullptr, num_splits, sl, ws + l.sws, l.sws_bytes,
      dtype, stream, &so_opts, &sin);
  if (st != PKV_OK) return st;
  if (pin.deferred) {
    cudaError_t e = launch_prefill_split_combine(
        pin.combine, pin.combine_max_q, pin.combine_bf16, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill split combine");
  }
  // with the overlap, the merge is a programmatic dependent of the last
  // suffix kernel, whose grid ends after the prefix grid
  cudaError_t e = launch_merge(output, po, pl, so, sl, nullptr, T, Hq, D,
                               dtype, dtype, s, overlap && !pin.deferred);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return PKV_OK;
}

pkv_status pkv_merge_attn_states(void* output, const void* prefix_output,
                                 const float* prefix_lse,
                                 const void* suffix_output,
                                 const float* suffix_lse, float* output_lse,
                                 int num_tokens, int num_heads, int head_size,
                                 pkv_dtype out_dtype, pkv_dtype in_dtype,
                                 pkv_stream_t stream) {
  if (num_tokens < 0 || num_heads <= 0 || head_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "bad sizes");
  if (head_size % 8 != 0 || head_size > 512)
    return fail(PKV_ERR_UNSUPPORTED,
                "head_size must be a multiple of 8 and at most 512");
  auto ok_dt = [](pkv_dtype d) {
    return d == PKV_F16 || d == PKV_BF16 || d == PKV_F32;
  };
  if (!ok_dt(out_dtype) || !ok_dt(in_dtype))
    return fail(PKV_ERR_UNSUPPORTED, "dtype must be fp16, bf16 or fp32");
  if ((out_dtype == PKV_F16 && in_dtype == PKV_BF16) ||
      (out_dtype == PKV_BF16 && in_dtype == PKV_F16))
    return fail(PKV_ERR_UNSUPPORTED, "fp16 and bf16 cannot be mixed");
  if (num_tokens == 0) return PKV_OK;
  if (!output || !prefix_output || !prefix_lse || !suffix_output ||
      !suffix_lse)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(output) || !aligned16(prefix_output) ||
      !aligned16(suffix_output))
    return fail(PKV_ERR_UNSUPPORTED, "outputs must be 16-byte aligned");
  cudaError_t e = launch_merge(output, prefix_output, prefix_lse,
                               suffix_output, suffix_lse, output_lse,
                               num_tokens, num_heads, head_size, out_dtype,
                               in_dtype, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return PKV_OK;
}

}  // extern "C"
