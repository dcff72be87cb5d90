// Persistent decode attention: every CTA streams an equal share of the
// batch's key tiles, for 16-bit and E4M3 (fp8) caches.
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (flash_attn_varlen_func over the paged cache: cu_seqlens_q,
// seqused_k, block_table, causal, window_size, softcap, alibi_slopes, LSE;
// kv_cache_dtype "fp8" with k_descale / v_descale) and
// FlashAttentionMetadataBuilder (split-KV decoding of requests with one
// query per KV-head group; partial results combined by their LSEs).
//
// Work order.  The decode-class requests (q_len * G <= 16 packed query rows
// per KV head) form a sequence of units u = b * Hkv + g (request b, KV head
// g), each a run of KT-key tiles over the unit's admissible key range: N
// tiles in all.  The launch is one wave of C CTAs, and the sequence is cut
// into C equal chunks, one per CTA, so every CTA moves the same number of
// K/V bytes whatever the spread of the request lengths (with one CTA per
// unit, the longest units of the last wave set the kernel's time).  A unit
// inside one chunk is finished there.  A unit that a chunk boundary cuts
// leaves one partial state (O normalised, LSE) per piece in the workspace,
// and fold_kernel merges the pieces by LSE.  (Measured on GB300: some SM
// groups stream K/V several percent slower than others, run after run, so
// equal chunks end a few microseconds apart; chunks dealt at run time from
// a ticket counter cost more in per-chunk start-up than they recovered.)
//
// CTA roles (NCW consumer warps + one producer warp):
//   producer   walks the CTA's units in order.  For each it publishes a
//              descriptor and cp.async-loads the unit's 16 packed query
//              rows into one of two Q slots (unit_full barrier), then
//              issues the unit's K and V page boxes with TMA into a
//              STAGES-deep ring, as the decode_tma kernel does.  It runs
//              ahead across unit boundaries, so the ring never drains
//              between units.
//   consumers  each own KT / NCW keys of every tile: S = Q K^T, online
//              softmax (base 2), O += P V on mma.sync m16n8k16.  At the end
//              of a unit the warps' states meet in the ring stage of the
//              unit's last tile, which stays held until they are merged,
//              and each warp normalises and writes a slice of the columns
//              (with D = 256, warp 0 merges all of them); the output, or
//              the piece's partial state.
//
// E4M3 caches.  The ring holds the codes (one byte per element, 128-column
// boxes).  The consumers convert them to f16 in registers with
// cvt.rn.f16x2.e4m3x2 (exact): K straight from an ldmatrix of the code
// bytes, V from an 8-bit transposing ldmatrix of the code bytes.
// The query rows are converted to f16 once per unit (a bf16 query is first
// scaled by a power of two that puts its largest magnitude in [2^14, 2^15),
// which keeps every value exact in f16; the factor joins the logit scale).
// The MMAs then run in f16, with the same key order in S and P V and a
// fixed permutation of the head dimension in S (the same for Q and K, so
// the dot products are unchanged).  k_scale joins the logit scale and
// v_scale multiplies the output.
//
// E4M3 queries (Q8, with an E4M3 cache).  The query rows arrive as codes,
// which convert exactly to the f16 fragments above (no scaling: every code
// is an f16 value), and q_scale joins the logit scale.  (The E4M3 form of
// mma.sync, m16n8k32, which would take the K code words as they are, was
// measured on GB300 at the same speed with 13 % more instructions issued,
// so the codes go through f16 like the cache's.)
//
// Every mbarrier wait is bounded (kWaitLimitNs).  A wait that runs out
// records kErrTimeout and raises the CTA's abort flag; the consumers agree
// on leaving at a barrier that reduces their flags (bar.red.or), and the
// producer drains the copies it issued before it exits.
#include <cuda.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pkv_common.cuh"
#include "tma_util.cuh"

namespace pkv {
namespace dsk {

constexpr int kMaxDevices = 64;
// Requests whose tile prefix a CTA keeps in shared memory (it locates its
// chunk there); larger batches locate it with one scan over the requests.
constexpr int kMaxPrefixReqs = 512;

template <int D, int NCW, int KT, int STAGES, bool KV8, bool Q8 = false>
struct Cfg {
  static constexpr int NT = (NCW + 1) * 32;     // consumers + producer warp
  static constexpr int CT = NCW * 32;           // consumer threads
  static constexpr int KW = KT / NCW;           // keys per warp per tile
  static constexpr int NKT = KW / 8;            // n8 tiles of S per warp
  static constexpr int BOXC = KV8 ? 128 : 64;   // columns per TMA box
  static constexpr int NCB = D / BOXC;          // 128-byte column blocks
  static constexpr int QEB = Q8 ? 1 : 2;       // bytes per query element
  static constexpr int CPR = D * QEB / 16;      // 16-byte chunks per Q row
  static constexpr int ROW_BYTES = D * QEB;     // one Q row
  static constexpr int CB_BYTES = KT * 128;     // one column block of a tile
  static constexpr int TILE_BYTES = NCB * CB_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int QRAW_BYTES = 16 * ROW_BYTES;
  static constexpr int QFRAG_BYTES = KV8 ? (D / 16) * 32 * 16 : 0;
  // The warps' states meet in the held stage of the unit's last tile: all
  // NCW of them when they fit (each warp then merges a column slice), else
  // those of warps 1.. (warp 0 merges with its own registers).
  static constexpr bool ALL_MERGE = NCW * 16 * D * 4 <= STAGE_BYTES;
  static constexpr int ML_BYTES = NCW * 16 * 2 * 4;
  static constexpr int PRE_BYTES = (kMaxPrefixReqs + 2) * 4;
  static constexpr int OFF_QRAW = RING_BYTES;
  static constexpr int OFF_QFRAG = OFF_QRAW + 2 * QRAW_BYTES;
  static constexpr int OFF_ML = OFF_QFRAG + QFRAG_BYTES;
  static constexpr int OFF_PRE = OFF_ML + ML_BYTES;
  static constexpr int OFF_DESC = OFF_PRE + PRE_BYTES;      // 2 x 64 bytes
  static constexpr int OFF_MISC = OFF_DESC + 128;           // 256 bytes
  static constexpr int OFF_BAR = OFF_MISC + 256;
  static constexpr int BAR_BYTES = (3 * STAGES + 4) * 8;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;   // + alignment
  static_assert(KW % 16 == 0, "each warp needs whole k16 steps of keys");
  static_assert(NKT == 2 || NKT == 4, "ldmatrix grouping of K");
  static_assert(D % BOXC == 0, "whole TMA boxes per row");
  static_assert(CB_BYTES % 1024 == 0, "128-byte swizzle atoms");
  static_assert(NCW >= 2, "several consumer warps");
  static_assert(ALL_MERGE || (NCW - 1) * 16 * D * 4 <= STAGE_BYTES,
                "the warps' states fit in one ring stage");
  static_assert((D / NCW) % 4 == 0, "column slices of whole float4s");
  static_assert(OFF_PRE % 8 == 0 && OFF_MISC % 8 == 0, "alignment");
  static_assert(!Q8 || KV8, "E4M3 queries need an E4M3 cache");
  static constexpr int KTILE = KT;
};

// Index of (row r, column col) of one warp's 16 x D state in the held
// stage; the column is XOR-swizzled by the row for conflict-free float2
// stores.
template <int D>
__device__ __forceinline__ int cidx(int r, int col) {
  return r * D + (col ^ ((r & 7) << 3));
}

// One unit piece as the producer hands it to the consumers (64 bytes).
struct UnitDesc {
  int b, g, q0, q_len;
  int rows, L, lo, hi;
  int kt0, t_beg, n_tiles, slot;   // slot: partial slot, or -1 (output)
  int end, pad0, pad1, pad2;       // end: no more units
};

// What a request contributes: its tile count per unit (0: not a
// decode-class request here) and its key geometry.
struct ReqInfo {
  int q0, q_len, rows, L, lo, hi, kt0, koff;
  int n_real;   // tiles over [kt0, hi)
  int n;        // tiles in the work sequence: max(n_real, 1), or 0
};

template <int KT>
__device__ __forceinline__ ReqInfo req_info(const AttnParams& p, int b,
                                            bool flag) {
  ReqInfo r{};
  r.q0 = p.cu_q[b];
  r.q_len = min(p.cu_q[b + 1] - r.q0, p.total_q - r.q0);
  if (r.q0 < 0 || r.q_len <= 0) return r;
  r.rows = r.q_len * p.G;
  if (r.rows < p.min_rows || r.rows > p.max_rows || r.rows > 16) return r;
  if (r.rows > p.sk_rows) {
    // more query rows than the call's max_seqlen_q allows (the partial
    // slots are sized by it): not computed, and reported
    if (flag) atomicOr(p.err, kErrQueryLen);
    return r;
  }
  r.koff = p.cu_k ? p.cu_k[b] : 0;
  r.L = p.cu_k ? p.cu_k[b + 1] - r.koff : p.seqused_k[b];
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  const int L_tab = p.cu_k ? (r.koff < 0 ? 0 : max(0, min(r.L, p.total_k - r.koff)))
                           : min(r.L, p.max_blocks * p.BS);
  if (flag && L_tab < r.L) atomicOr(p.err, kErrBadTable);
  int kmin, kmax;
  key_range(r.L, r.q_len, 0, r.q_len - 1, p.causal, p.wl, p.wr, kmin, kmax);
  r.lo = kmin;
  r.hi = max(kmin, min(kmax, L_tab));
  r.kt0 = (r.lo / KT) * KT;
  r.n_real = r.hi > r.lo ? (r.hi - r.kt0 + KT - 1) / KT : 0;
  r.n = max(r.n_real, 1);
  return r;
}

// Byte offset of 16-byte chunk `ch` (0 .. D*EB/16-1) of row r in a tile
// written by 128-byte-wide TMA boxes with the 128-byte swizzle.
template <int KT>
__device__ __forceinline__ uint32_t kv_off(int r, int ch) {
  return static_cast<uint32_t>((ch >> 3) * (KT * 128)) + sw128(r, ch & 7);
}

// All consumer threads reach named barrier 1; returns the OR of `pred`.
__device__ __forceinline__ bool bar_or(int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(n)
               : "memory");
}

__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}


template <typename T, int D, int NCW, int KT, int STAGES, bool KV8, bool Q8>
__global__ void __launch_bounds__((NCW + 1) * 32, 2)
decode_sk_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<D, NCW, KT, STAGES, KV8, Q8>;
  // MMA input type: the cache's type, or f16 for E4M3 codes
  using MT = typename std::conditional<KV8, __half, T>::type;
  // launched as a programmatic dependent of the kernel before it: the CTAs
  // are resident while that kernel ends; nothing is read before it is
  // complete and its writes are visible (a no-op for a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_u - raw_u);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int Hkv = p.Hkv, G = p.G;

  const uint32_t ring = base_u;
  const uint32_t bar0 = base_u + C::OFF_BAR;
  auto full_k = [&](int s) { return bar0 + 8 * s; };
  auto full_v = [&](int s) { return bar0 + 8 * (STAGES + s); };
  auto empty = [&](int s) { return bar0 + 8 * (2 * STAGES + s); };
  auto ufull = [&](int s) { return bar0 + 8 * (3 * STAGES + s); };
  auto uempty = [&](int s) { return bar0 + 8 * (3 * STAGES + 2 + s); };
  auto tile_k = [&](int s) { return ring + s * C::STAGE_BYTES; };
  auto tile_v = [&](int s) {
    return ring + s * C::STAGE_BYTES + C::TILE_BYTES;
  };
  auto qraw = [&](int s) { return base_u + C::OFF_QRAW + s * C::QRAW_BYTES; };
  const uint32_t qfrag = base_u + C::OFF_QFRAG;
  float* ml = reinterpret_cast<float*>(base + C::OFF_ML);
  int* pre = reinterpret_cast<int*>(base + C::OFF_PRE);
  volatile UnitDesc* desc =
      reinterpret_cast<volatile UnitDesc*>(base + C::OFF_DESC);
  int* misc = reinterpret_cast<int*>(base + C::OFF_MISC);
  volatile int* abort_flag = misc;                 // [0]
  volatile unsigned* bad_boxes =
      reinterpret_cast<volatile unsigned*>(misc + 1);   // [1 .. STAGES]
  int* start = misc + 8;                           // [8 .. 15]
  long long* scan = reinterpret_cast<long long*>(misc + 16);   // [16 .. 31]
  float* qmax = reinterpret_cast<float*>(misc + 32);            // [32 .. 39]

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_k(s), 1);
      mbar_init(full_v(s), 1);
      mbar_init(empty(s), NCW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(ufull(s), 1 + 32);   // descriptor + the producer's cp.asyncs
      mbar_init(uempty(s), NCW);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- the tile sequence (every CTA derives the same prefix over the
  // requests; thread t scans a contiguous run of them)
  const int B = p.batch;
  const int per = (B + C::NT - 1) / C::NT;
  const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
  // (the fold kernel may start: it waits for this grid before reading)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  long long mine = 0;
  for (int b = b_lo; b < b_hi; ++b) {
    const long long n =
        static_cast<long long>(req_info<KT>(p, b, c == 0).n) * Hkv;
    mine += n;
    if (B <= kMaxPrefixReqs) pre[b] = static_cast<int>(n);  // (kept below
  }                                                          // if N fits)
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  long long excl = incl - mine, N = 0;
  for (int w = 0; w < NCW + 1; ++w) {
    if (w < warp) excl += scan[w];
    N += scan[w];
  }
  // the per-request prefix in shared memory (small batches): any CTA can
  // then locate any chunk
  const bool table = B <= kMaxPrefixReqs && N < (1LL << 30);
  if (table) {
    long long acc = excl;
    for (int b = b_lo; b < b_hi; ++b) {
      const int n = pre[b];
      pre[b] = static_cast<int>(acc);
      acc += n;
    }
    if (tid == 0) pre[B] = static_cast<int>(N);
  }

  // ---- chunks: Cs equal ones, one per CTA, at least two tiles each (every
  // chunk holds a tile: the fold follows a unit's pieces through
  // consecutive chunks)
  const int C_all = gridDim.x;
  const long long Cs = max(1LL, min(static_cast<long long>(C_all), N / 2));
  auto bound = [&](long long k) -> long long { return k * N / Cs; };
  if (c >= Cs && tid == 0) p.sk_marks[c] = make_int2(-1, -1);
  if (!table && c < Cs) {
    // the CTA's static chunk located by the thread whose run holds it
    const long long T0 = bound(c), T1 = bound(c + 1);
    if (T0 < T1 && mine > 0) {
      long long acc = excl;
      for (int b = b_lo; b < b_hi; ++b) {
        const int n = req_info<KT>(p, b, false).n;
        const long long t = static_cast<long long>(n) * Hkv;
        if (n > 0) {
          if (T0 >= acc && T0 < acc + t) {
            start[0] = b;
            start[1] = static_cast<int>((T0 - acc) / n);
            start[2] = static_cast<int>((T0 - acc) % n);
            start[7] = n;
          }
          if (T1 - 1 >= acc && T1 - 1 < acc + t) {
            start[3] = b;
            start[4] = static_cast<int>((T1 - 1 - acc) / n);
            start[5] = static_cast<int>((T1 - 1 - acc) % n);
            start[6] = n;
          }
        }
        acc += t;
      }
    }
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    constexpr int CPR = C::CPR;
    const int RB = p.rb;
    const int nb_max = KT / RB;
    const char* Q = static_cast<const char*>(p.q);
    // K/V pages are read once: their L2 lines go first
    const uint64_t pol = l2_evict_first_policy();
    // (request, KV head, tile) of tile position P of the sequence
    auto locate = [&](long long P, int& b, int& g, int& t, int& n) {
      int lo = 0, hi = B;          // pre[lo] <= P < pre[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= P) lo = mid; else hi = mid;
      }
      b = lo;
      n = (pre[lo + 1] - pre[lo]) / Hkv;
      const int rel = static_cast<int>(P - pre[lo]);
      g = rel / n;
      t = rel - g * n;
    };
    int k = 0, it = 0;
    bool stop = false;
    const long long chunk = c;
    if (c < Cs) {
      const long long T0 = bound(chunk), T1 = bound(chunk + 1);
      int b, g, t, n0, b1, g1, t1, n1;
      if (table) {
        locate(T0, b, g, t, n0);
        locate(T1 - 1, b1, g1, t1, n1);
      } else {
        b = start[0]; g = start[1]; t = start[2]; n0 = start[7];
        b1 = start[3]; g1 = start[4]; t1 = start[5]; n1 = start[6];
      }
      (void)n0;
      // pieces left for the fold: the unit the chunk starts inside (head,
      // slot 2 chunk) and the unit it starts that runs past its end (tail,
      // slot 2 chunk + 1)
      const int u0 = b * Hkv + g, u1 = b1 * Hkv + g1;
      const int head_u = t > 0 ? u0 : -1;
      const int tail_u = (t1 + 1 < n1 && !(u1 == u0 && t > 0)) ? u1 : -1;
      if (lane == 0) p.sk_marks[chunk] = make_int2(head_u, tail_u);

      long long pos = T0;
      ReqInfo ri = req_info<KT>(p, b, false);
      while (pos < T1) {
        const int slot = k & 1;
        if (k >= 2) {
          int ok = 1;
          if (lane == 0)
            ok = mbar_wait_lim(uempty(slot), ((k >> 1) - 1) & 1, abort_flag,
                        p.err, p.wait_ns);
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            stop = true;
            break;
          }
        }
        const long long len =
            min(static_cast<long long>(ri.n - t), T1 - pos);
        int pslot = -1;
        if (pos == T0 && head_u >= 0)
          pslot = 2 * static_cast<int>(chunk);
        else if (pos + len == T1 && tail_u >= 0)
          pslot = 2 * static_cast<int>(chunk) + 1;
        const int j_beg = t;
        const int j_end = min(t + static_cast<int>(len), ri.n_real);
        if (lane == 0) {
          volatile UnitDesc& d = desc[slot];
          d.b = b;
          d.g = g;
          d.q0 = ri.q0;
          d.q_len = ri.q_len;
          d.rows = ri.rows;
          d.L = ri.L;
          d.lo = ri.lo;
          d.hi = ri.hi;
          d.kt0 = ri.kt0;
          d.t_beg = j_beg;
          d.n_tiles = max(0, j_end - j_beg);
          d.slot = pslot;
          d.end = 0;
        }
        // the unit's 16 packed query rows (zeros past `rows`)
        for (int i = lane; i < 16 * CPR; i += 32) {
          const int r = i / CPR, ch = i - (i / CPR) * CPR;
          const bool ok = r < ri.rows;
          const char* src = Q;
          if (ok)
            src = Q + (static_cast<int64_t>(ri.q0 + r / G) * p.q_st +
                       static_cast<int64_t>(g * G + r % G) * p.q_sh) *
                          C::QEB +
                  ch * 16;
          cp_async_16(qraw(slot) + swz<C::ROW_BYTES>(r, ch), src,
                      ok ? 16 : 0);
        }
        if (lane == 0) mbar_arrive(ufull(slot));
        cp_async_mbar_arrive(ufull(slot));

        // the piece's K and V tiles
        const int32_t* bt =
            p.cu_k ? nullptr
                   : p.block_table + static_cast<int64_t>(b) * p.bt_stride;
        auto fetch = [&](int j) -> int {          // page id of box `lane`
          const int k0 = ri.kt0 + j * KT + lane * RB;
          if (j >= j_end || lane >= nb_max || k0 >= ri.hi || !bt) return 0;
          const int blk = __ldg(bt + k0 / p.BS);
          if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(p.err, kErrBadBlock);
            return -1;
          }
          return blk;
        };
        int cur = fetch(j_beg);
        for (int j = j_beg; j < j_end; ++j) {
          const int nxt = fetch(j + 1);
          const int s = it % STAGES;
          const int kt = ri.kt0 + j * KT;
          int nbox = (ri.hi - kt + RB - 1) / RB;
          if (nbox > nb_max) nbox = nb_max;
          const unsigned bad =
              __ballot_sync(0xffffffffu, lane < nbox && cur < 0);
          int halt = 0;
          if (lane == 0) {
            if (it >= STAGES &&
                !mbar_wait_lim(empty(s), ((it / STAGES) - 1) & 1, abort_flag,
                        p.err, p.wait_ns)) {
              halt = 1;
            } else {
              bad_boxes[s] = bad;
              const uint32_t bytes =
                  (nbox - __popc(bad)) * C::NCB * RB * 128;
              mbar_expect_tx(full_k(s), bytes);
              mbar_expect_tx(full_v(s), bytes);
            }
          }
          if (__shfl_sync(0xffffffffu, halt, 0)) {
            stop = true;
            break;
          }
          if (lane < nbox && cur >= 0) {
            const int k0 = kt + lane * RB;
            const int row = p.cu_k ? ri.koff + k0 : k0 % p.BS;
#pragma unroll
            for (int cb = 0; cb < C::NCB; ++cb) {
              const uint32_t dk =
                  tile_k(s) + cb * C::CB_BYTES + lane * RB * 128;
              const uint32_t dv =
                  tile_v(s) + cb * C::CB_BYTES + lane * RB * 128;
              if (p.kv_order_hnd) {
                tma_load_4d_hint(dk, &tm_k, cb * C::BOXC, row, g, cur,
                                 full_k(s), pol);
                tma_load_4d_hint(dv, &tm_v, cb * C::BOXC, row, g, cur,
                                 full_v(s), pol);
              } else {
                tma_load_4d_hint(dk, &tm_k, cb * C::BOXC, g, row, cur,
                                 full_k(s), pol);
                tma_load_4d_hint(dv, &tm_v, cb * C::BOXC, g, row, cur,
                                 full_v(s), pol);
              }
            }
          }
          ++it;
          cur = nxt;
        }
        if (stop) break;
        pos += len;
        ++k;
        if (pos < T1) {
          t = 0;
          if (++g == Hkv) {
            g = 0;
            do {
              ++b;
              ri = req_info<KT>(p, b, false);
            } while (ri.n == 0 && b + 1 < B);
            if (ri.n == 0) pos = T1;    // (unreachable: the scan saw tiles)
          }
        }
      }
    }
    if (!stop) {
      // no more units: publish the end of the sequence
      const int slot = k & 1;
      int ok = 1;
      if (k >= 2 && lane == 0)
        ok = mbar_wait_lim(uempty(slot), ((k >> 1) - 1) & 1, abort_flag,
                        p.err, p.wait_ns);
      if (__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          desc[slot].end = 1;
          mbar_arrive(ufull(slot));
        }
        cp_async_mbar_arrive(ufull(slot));
      }
    }
    if (lane == 0) {
      // no copy of this CTA may still be in flight when it exits
      for (int j = max(0, it - STAGES); j < it; ++j) {
        mbar_drain(full_k(j % STAGES), (j / STAGES) & 1);
        mbar_drain(full_v(j % STAGES), (j / STAGES) & 1);
      }
    }
    cp_async_wait<0>();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g8 = lane >> 2, c4 = lane & 3;
  const int rA = g8, rB = g8 + 8;
  const int lm_mi = lane >> 3, lm_r = lane & 7;
  const int kw0 = warp * C::KW;
  const bool plain = (p.softcap <= 0.f) && (p.alibi == nullptr);
  const bool capped = (p.softcap > 0.f) && (p.alibi == nullptr);
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
  const float vscale = p.v_scale ? *p.v_scale : 1.f;
  const float kscale = p.k_scale ? *p.k_scale : 1.f;
  const float qscale = Q8 ? *p.q_scale : 1.f;
  T* __restrict__ OUT = static_cast<T*>(p.out);
  int it = 0;

  for (int k = 0;; ++k) {
    const int slot = k & 1;
    const bool got = mbar_wait_lim(ufull(slot), (k >> 1) & 1, abort_flag,
                        p.err, p.wait_ns);
    float qshift_f = 1.f;    // 2^shift: the query scaling of an fp8 unit
    if constexpr (Q8) {
      if (bar_or(C::CT, !got)) return;
      // f16 A fragments of the codes for every k16 step, in the order of
      // the 16-bit query path below (d = 16 ks + 4 c + {0,1} in registers
      // 0/1, + {2,3} in registers 2/3; rows g and g + 8)
      for (int i = tid; i < (D / 16) * 32; i += C::CT) {
        const int ks = i >> 5, ln = i & 31;
        const int gg = ln >> 2, cc = ln & 3;
        const int d = 16 * ks + 4 * cc;
        uint32_t a[4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          e4m3x4_to_f16(lds32(qraw(slot) +
                              swz<C::ROW_BYTES>(gg + 8 * h, d >> 4) + (d & 15)),
                        a[h], a[2 + h]);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         qfrag + (ks * 32 + ln) * 16),
                     "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3])
                     : "memory");
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");
    } else if constexpr (KV8) {
      // largest |q| of the unit's rows (bf16 queries only)
      float mx = 0.f;
      if (got && std::is_same<T, __nv_bfloat16>::value) {
        for (int i = tid; i < 16 * C::CPR; i += C::CT) {
          const int r = i / C::CPR, ch = i - (i / C::CPR) * C::CPR;
          uint32_t w[4];
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qraw(slot) + swz<C::ROW_BYTES>(r, ch)));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            mx = fmaxf(mx, fabsf(elem_f32<T>(w[e], 0)));
            mx = fmaxf(mx, fabsf(elem_f32<T>(w[e], 1)));
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) qmax[warp] = mx;
      }
      if (bar_or(C::CT, !got)) return;
      int shift = 0;
      if (std::is_same<T, __nv_bfloat16>::value) {
        float m = 0.f;
        for (int w = 0; w < NCW; ++w) m = fmaxf(m, qmax[w]);
        if (m > 0.f) {
          const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xff) - 127;
          shift = max(-100, min(100, e - 14));
        }
      }
      qshift_f = exp2f(static_cast<float>(shift));
      const float qmul = exp2f(static_cast<float>(-shift));
      // f16 A fragments of Q for every k16 step, in the head-dimension
      // order the K fragments arrive in (d = 16 ks + 4 c4 + {0,1} in
      // registers 0/1, + {2,3} in registers 2/3)
      for (int i = tid; i < (D / 16) * 32; i += C::CT) {
        const int ks = i >> 5, ln = i & 31;
        const int gg = ln >> 2, cc = ln & 3;
        const int d = 16 * ks + 4 * cc;
        const uint32_t off = (d & 7) * 2;
        uint32_t a[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w0, w1;
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                       : "=r"(w0), "=r"(w1)
                       : "r"(qraw(slot) + swz<C::ROW_BYTES>(gg + 8 * h, d >> 3) +
                             off));
          if (std::is_same<T, __half>::value) {
            a[h] = w0;
            a[2 + h] = w1;
          } else {
            a[h] = pack2<__half>(elem_f32<T>(w0, 0) * qmul,
                                 elem_f32<T>(w0, 1) * qmul);
            a[2 + h] = pack2<__half>(elem_f32<T>(w1, 0) * qmul,
                                     elem_f32<T>(w1, 1) * qmul);
          }
        }
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         qfrag + (ks * 32 + ln) * 16),
                     "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3])
                     : "memory");
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");
    } else {
      if (bar_or(C::CT, !got)) return;
    }
    const int d_end = desc[slot].end;
    if (d_end) return;
    const int b = desc[slot].b, g = desc[slot].g, q0 = desc[slot].q0;
    const int q_len = desc[slot].q_len, rows = desc[slot].rows;
    const int L = desc[slot].L, lo = desc[slot].lo, hi = desc[slot].hi;
    const int kt0 = desc[slot].kt0, t_beg = desc[slot].t_beg;
    const int n_tiles = desc[slot].n_tiles, pslot = desc[slot].slot;
    (void)b;
    if constexpr (KV8) {
      // Q now lives in the fragment buffer: release the descriptor slot
      __syncwarp();
      if (lane == 0) mbar_arrive(uempty(slot));
    }

    const int ctx = L - q_len;
    const int pA = ctx + rA / G, pB = ctx + rB / G;
    const bool okA = rA < rows, okB = rB < rows;
    float slopeA = 0.f, slopeB = 0.f;
    if (p.alibi) {
      if (okA) slopeA = p.alibi[g * G + rA % G];
      if (okB) slopeB = p.alibi[g * G + rB % G];
    }
    const float qk_scale = p.scale * kscale * qshift_f * qscale;
    const float scale_log2 = qk_scale * kLog2e;
    int full_lo = lo, full_hi = hi;
    {
      const int p_lo = ctx, p_hi = ctx + (rows - 1) / G;
      if (p.wl >= 0) full_lo = max(full_lo, p_hi - p.wl);
      if (p.causal) full_hi = min(full_hi, p_lo + 1);
      if (p.wr >= 0) full_hi = min(full_hi, p_lo + p.wr + 1);
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    bool aborted = false;

    for (int jt = 0; jt < n_tiles; ++jt, ++it) {
      const int s = it % STAGES;
      const uint32_t par = (it / STAGES) & 1;
      const int kt = kt0 + (t_beg + jt) * KT;
      if (!mbar_wait_lim(full_k(s), par, abort_flag,
                        p.err, p.wait_ns)) {
        aborted = true;
        break;
      }
      const uint32_t sK = tile_k(s), sV = tile_v(s);
      constexpr int RCH = KV8 ? D / 16 : D / 8;   // 16-byte chunks per row
      if (const unsigned bad = bad_boxes[s]) {
        // pages the table pointed outside the cache: zero keys and values
        for (int idx = lane; idx < C::KW * RCH; idx += 32) {
          const int r = kw0 + idx / RCH, ch = idx % RCH;
          if (!((bad >> (r / p.rb)) & 1u)) continue;
          asm volatile("st.shared.v4.u32 [%0], {%2, %2, %2, %2};\n"
                       "st.shared.v4.u32 [%1], {%2, %2, %2, %2};" ::"r"(
                           sK + kv_off<KT>(r, ch)),
                       "r"(sV + kv_off<KT>(r, ch)), "r"(0)
                       : "memory");
        }
        fence_proxy_async();
        __syncwarp();
      }

      // S = Q K^T for 16 rows x KW keys
      float sc[C::NKT][4];
#pragma unroll
      for (int i = 0; i < C::NKT; ++i)
        sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      if constexpr (KV8) {
        // one ldmatrix.x4 group holds 4 / NKT k16 steps of all NKT n8
        // tiles: matrix m covers n8 tile m % NKT of step grp * 4 / NKT +
        // m / NKT (16 code bytes = one k16 step)
        constexpr int KPG = 4 / C::NKT;
#pragma unroll
        for (int grp = 0; grp < (D / 16) / KPG; ++grp) {
          uint32_t r4[4];
          {
            const int nt = lm_mi % C::NKT, ks = grp * KPG + lm_mi / C::NKT;
            ldmatrix_x4(sK + kv_off<KT>(kw0 + nt * 8 + lm_r, ks), r4[0],
                        r4[1], r4[2], r4[3]);
          }
#pragma unroll
          for (int kq = 0; kq < KPG; ++kq) {
            const int ks = grp * KPG + kq;
            uint32_t a[4];
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                         : "r"(qfrag + (ks * 32 + lane) * 16));
#pragma unroll
            for (int nt = 0; nt < C::NKT; ++nt) {
              uint32_t b0, b1;
              e4m3x4_to_f16(r4[kq * C::NKT + nt], b0, b1);
              mma_16816<__half>(sc[nt], a, b0, b1);
            }
          }
        }
      } else {
        const uint32_t sQ = qraw(slot);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4];
          {
            const int r = lm_r + (lm_mi & 1) * 8;
            const int ch = kk * 2 + (lm_mi >> 1);
            ldmatrix_x4(sQ + swz<C::ROW_BYTES>(r, ch), a[0], a[1], a[2], a[3]);
          }
#pragma unroll
          for (int np = 0; np < C::NKT / 2; ++np) {
            uint32_t b0, b1, b2, b3;
            const int r = kw0 + np * 16 + lm_r + (lm_mi >> 1) * 8;
            const int ch = kk * 2 + (lm_mi & 1);
            ldmatrix_x4(sK + kv_off<KT>(r, ch), b0, b1, b2, b3);
            mma_16816<T>(sc[2 * np], a, b0, b1);
            mma_16816<T>(sc[2 * np + 1], a, b2, b3);
          }
        }
      }

      // logits (base 2) with masks
      float mxA = -INFINITY, mxB = -INFINITY;
      const bool interior = kt >= full_lo && kt + KT <= full_hi;
      if (plain && interior) {
#pragma unroll
        for (int nt = 0; nt < C::NKT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] *= scale_log2;
          mxA = fmaxf(mxA, fmaxf(sc[nt][0], sc[nt][1]));
          mxB = fmaxf(mxB, fmaxf(sc[nt][2], sc[nt][3]));
        }
      } else if (capped && interior) {
        const float pre = qk_scale * inv_cap, post = p.softcap * kLog2e;
#pragma unroll
        for (int nt = 0; nt < C::NKT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sc[nt][e] = post * tanh_fast(sc[nt][e] * pre);
          mxA = fmaxf(mxA, fmaxf(sc[nt][0], sc[nt][1]));
          mxB = fmaxf(mxB, fmaxf(sc[nt][2], sc[nt][3]));
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < C::NKT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = kt + kw0 + nt * 8 + 2 * c4 + (e & 1);
            const bool rowB = e >= 2;
            const int pos = rowB ? pB : pA;
            float x = sc[nt][e];
            if (plain) {
              x *= scale_log2;
            } else {
              x *= qk_scale;
              if (p.softcap > 0.f) x = p.softcap * tanh_fast(x * inv_cap);
              if (p.alibi)
                x -= (rowB ? slopeB : slopeA) * fabsf(float(pos - key));
              x *= kLog2e;
            }
            bool ok = (rowB ? okB : okA) && key >= lo && key < hi;
            if (p.causal) ok = ok && key <= pos;
            if (p.wl >= 0) ok = ok && key >= pos - p.wl;
            if (p.wr >= 0) ok = ok && key <= pos + p.wr;
            x = ok ? x : -INFINITY;
            sc[nt][e] = x;
            if (rowB) mxB = fmaxf(mxB, x); else mxA = fmaxf(mxA, x);
          }
        }
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
      const float baseA = (mnA == -INFINITY) ? 0.f : mnA;
      const float baseB = (mnB == -INFINITY) ? 0.f : mnB;
      const float alA = ex2(mA - baseA), alB = ex2(mB - baseB);
      mA = mnA;
      mB = mnB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int nt = 0; nt < C::NKT; ++nt) {
        sc[nt][0] = ex2(sc[nt][0] - baseA);
        sc[nt][1] = ex2(sc[nt][1] - baseA);
        sc[nt][2] = ex2(sc[nt][2] - baseB);
        sc[nt][3] = ex2(sc[nt][3] - baseB);
        sumA += sc[nt][0] + sc[nt][1];
        sumB += sc[nt][2] + sc[nt][3];
      }
      lA = lA * alA + sumA;
      lB = lB * alB + sumB;
      // once the running maxima settle, alpha is exactly 1: skip the rescale
      if (__any_sync(0xffffffffu, alA != 1.f || alB != 1.f)) {
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o[i][0] *= alA;
          o[i][1] *= alA;
          o[i][2] *= alB;
          o[i][3] *= alB;
        }
      }

      if (!mbar_wait_lim(full_v(s), par, abort_flag,
                        p.err, p.wait_ns)) {
        aborted = true;
        break;
      }
      if (kt + kw0 + C::KW > hi) {
        // rows of this warp at or past the loaded range: zero them, so
        // that P = 0 never meets NaN padding or a stale row
        const int r0 = max(hi - kt, kw0);
        for (int idx = lane; idx < (kw0 + C::KW - r0) * RCH; idx += 32) {
          const int r = r0 + idx / RCH, ch = idx % RCH;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                           sV + kv_off<KT>(r, ch)),
                       "r"(0)
                       : "memory");
        }
        fence_proxy_async();
        __syncwarp();
      }
      // O += P V
#pragma unroll
      for (int ks = 0; ks < C::KW / 16; ++ks) {
        uint32_t a[4];
        a[0] = pack2<MT>(sc[2 * ks][0], sc[2 * ks][1]);
        a[1] = pack2<MT>(sc[2 * ks][2], sc[2 * ks][3]);
        a[2] = pack2<MT>(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
        a[3] = pack2<MT>(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
        if constexpr (KV8) {
          // V^T fragments straight from the code bytes: the 8-bit
          // transposing ldmatrix of a 16-key x 16-column block gives each
          // lane four keys of column g8 (d0) and of column g8 + 8 (d1).
          // The row addresses take the keys in the order 2c, 2c + 1,
          // 2c + 8, 2c + 9 (c = 0 .. 3), so a lane's four are the B
          // fragment's k = 2 c4, 2 c4 + 1, 2 c4 + 8, 2 c4 + 9.
          const int li = lane & 15;
          const int kr = kw0 + ks * 16 + 2 * (li >> 2) + (li & 1) +
                         ((li & 2) ? 8 : 0);
#pragma unroll
          for (int q = 0; q < D / 16; ++q) {
            uint32_t d0, d1, b0, b1, b2, b3;
            ldmatrix_b8_trans(sV + kv_off<KT>(kr, q), d0, d1);
            e4m3x4_to_f16(d0, b0, b1);
            e4m3x4_to_f16(d1, b2, b3);
            mma_16816<__half>(o[2 * q], a, b0, b1);
            mma_16816<__half>(o[2 * q + 1], a, b2, b3);
          }
        } else {
#pragma unroll
          for (int dp = 0; dp < D / 16; ++dp) {
            uint32_t b0, b1, b2, b3;
            const int r = kw0 + ks * 16 + lm_r + (lm_mi & 1) * 8;
            const int ch = dp * 2 + (lm_mi >> 1);
            ldmatrix_x4_trans(sV + kv_off<KT>(r, ch), b0, b1, b2, b3);
            mma_16816<T>(o[2 * dp], a, b0, b1);
            mma_16816<T>(o[2 * dp + 1], a, b2, b3);
          }
        }
      }
      __syncwarp();
      // the unit's last stage stays held: the epilogue merges in it
      if (lane == 0 && jt + 1 < n_tiles) mbar_arrive(empty(s));
    }
    if constexpr (!KV8) {
      // the unit's Q slot and descriptor are no longer read
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(uempty(slot));
    }

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);

    // ---- epilogue: the warps' states meet in the held stage of the unit's
    // last tile (a unit without tiles has nothing to merge: every warp's
    // state is empty and warp 0 writes the empty row)
    if (bar_or(C::CT, aborted || *abort_flag)) return;
    const int held = (it + STAGES - 1) % STAGES;
    float* comb = reinterpret_cast<float*>(base + (tile_k(held) - base_u));
    const float* sinks = pslot < 0 ? p.sinks : nullptr;  // once, here or in
                                                         // the fold
    auto store_row = [&](int r, int col, float4 v, float inv, float lse) {
      const int tok = q0 + r / G, hq = g * G + r % G;
      if (pslot < 0) {
        T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
                 static_cast<int64_t>(hq) * p.o_sh + col;
        uint2 pk;
        pk.x = pack2<T>(v.x * inv, v.y * inv);
        pk.y = pack2<T>(v.z * inv, v.w * inv);
        *reinterpret_cast<uint2*>(dst) = pk;
        if (col == 0 && p.lse)
          p.lse[static_cast<int64_t>(hq) * p.total_q + tok] = lse;
      } else {
        const int64_t sr = static_cast<int64_t>(pslot) * p.sk_rows + r;
        *reinterpret_cast<float4*>(p.part_o + sr * D + col) =
            make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        if (col == 0) p.part_lse[sr] = lse;
      }
    };
    if (n_tiles == 0) {
      if (warp == 0) {
        for (int i = lane; i < rows * (D / 4); i += 32) {
          const int r = i / (D / 4), col = (i - r * (D / 4)) * 4;
          float inv, lse;
          finish_row(-INFINITY, 0.f, sinks, g * G + r % G, &inv, &lse);
          store_row(r, col, make_float4(0.f, 0.f, 0.f, 0.f), 0.f, lse);
        }
      }
      continue;
    }
    // this warp's state into the stage (all warps, or warps 1..)
    const int wslot = C::ALL_MERGE ? warp : warp - 1;
    if (wslot >= 0) {
      float* cw = comb + wslot * 16 * D;
      if (c4 == 0) {
        ml[wslot * 32 + rA * 2] = mA;
        ml[wslot * 32 + rA * 2 + 1] = lA;
        ml[wslot * 32 + rB * 2] = mB;
        ml[wslot * 32 + rB * 2 + 1] = lB;
      }
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        *reinterpret_cast<float2*>(cw + cidx<D>(rA, dn * 8 + 2 * c4)) =
            make_float2(o[dn][0], o[dn][1]);
        *reinterpret_cast<float2*>(cw + cidx<D>(rB, dn * 8 + 2 * c4)) =
            make_float2(o[dn][2], o[dn][3]);
      }
      fence_proxy_async();   // the producer's TMA rewrites this stage later
    }
    asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");

    if constexpr (C::ALL_MERGE) {
      // every warp merges, normalises and writes one column slice
      constexpr int CW4 = D / NCW / 4;
      for (int i = lane; i < rows * CW4; i += 32) {
        const int r = i / CW4;
        const int col = warp * (D / NCW) + (i - r * CW4) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[w * 32 + r * 2]);
        const float mb = (M == -INFINITY) ? 0.f : M;
        float lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float f = ex2(ml[w * 32 + r * 2] - mb);
          lsum += f * ml[w * 32 + r * 2 + 1];
          const float4 v = *reinterpret_cast<const float4*>(
              comb + w * 16 * D + cidx<D>(r, col));
          acc.x += f * v.x;
          acc.y += f * v.y;
          acc.z += f * v.z;
          acc.w += f * v.w;
        }
        float inv, lse;
        finish_row(M, lsum, sinks, g * G + r % G, &inv, &lse);
        store_row(r, col, acc, inv * vscale, lse);
      }
      // the held stage goes back to the producer (one arrival per warp)
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(held));
    } else {
      if (warp != 0) continue;
      // warp 0 merges the others' states into its registers' rows
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = g8 + 8 * h;
        if (r >= rows) continue;
        const float m_own = h ? mB : mA, l_own = h ? lB : lA;
        float M = m_own;
#pragma unroll
        for (int w = 0; w < NCW - 1; ++w) M = fmaxf(M, ml[w * 32 + r * 2]);
        const float mb = (M == -INFINITY) ? 0.f : M;
        const float f_own = ex2(m_own - mb);
        float fw[NCW - 1];
        float lsum = f_own * l_own;
#pragma unroll
        for (int w = 0; w < NCW - 1; ++w) {
          fw[w] = ex2(ml[w * 32 + r * 2] - mb);
          lsum += fw[w] * ml[w * 32 + r * 2 + 1];
        }
        float inv, lse;
        finish_row(M, lsum, sinks, g * G + r % G, &inv, &lse);
        inv *= vscale;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          const int col = dn * 8 + 2 * c4;
          float v0 = f_own * o[dn][2 * h], v1 = f_own * o[dn][2 * h + 1];
#pragma unroll
          for (int w = 0; w < NCW - 1; ++w) {
            const float2 x = *reinterpret_cast<const float2*>(
                comb + w * 16 * D + cidx<D>(r, col));
            v0 += fw[w] * x.x;
            v1 += fw[w] * x.y;
          }
          const int tok = q0 + r / G, hq = g * G + r % G;
          if (pslot < 0) {
            *reinterpret_cast<uint32_t*>(
                OUT + static_cast<int64_t>(tok) * p.o_st +
                static_cast<int64_t>(hq) * p.o_sh + col) =
                pack2<T>(v0 * inv, v1 * inv);
            if (col == 0 && p.lse)
              p.lse[static_cast<int64_t>(hq) * p.total_q + tok] = lse;
          } else {
            const int64_t sr = static_cast<int64_t>(pslot) * p.sk_rows + r;
            *reinterpret_cast<float2*>(p.part_o + sr * D + col) =
                make_float2(v0 * inv, v1 * inv);
            if (col == 0) p.part_lse[sr] = lse;
          }
        }
      }
      // the held stage goes back to the producer (for all NCW warps)
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive_n(empty(held), NCW);
    }
  }
}

// Merge the pieces of the units that chunk boundaries cut.  Block c
// (1 <= c < chunks) looks at the boundary before chunk c: the unit whose
// first piece chunk c - 1 wrote to slot 2(c-1)+1 continues in slots 2c,
// 2(c+1), ... for every following chunk that marks it as its head unit.
template <typename T, int D>
__global__ void __launch_bounds__(128) fold_kernel(const AttnParams p,
                                                   int chunks) {
  // a prefill launch queued after this one in the same call may start
  // before this grid ends (it writes other requests' rows)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // launched as a programmatic dependent of the decode grid: wait until it
  // has finished and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c = blockIdx.x + 1;
  const int u = p.sk_marks[c - 1].y;
  if (u < 0) return;
  int c_end = c;
  while (c_end < chunks && p.sk_marks[c_end].x == u) ++c_end;
  const int npieces = 1 + (c_end - c);
  const int b = u / p.Hkv, g = u - (u / p.Hkv) * p.Hkv;
  const int q0 = p.cu_q[b];
  const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
  const int rows = min(q_len * p.G, p.sk_rows);
  T* __restrict__ OUT = static_cast<T*>(p.out);
  auto slot_of = [&](int k) {
    return k == 0 ? 2 * (c - 1) + 1 : 2 * (c + k - 1);
  };
  for (int i = threadIdx.x; i < rows * (D / 4); i += blockDim.x) {
    const int r = i / (D / 4), col = (i - r * (D / 4)) * 4;
    float M = -INFINITY;
    for (int k = 0; k < npieces; ++k)
      M = fmaxf(M, p.part_lse[static_cast<int64_t>(slot_of(k)) * p.sk_rows + r] *
                       kLog2e);
    const float mb = (M == -INFINITY) ? 0.f : M;
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < npieces; ++k) {
      const int64_t sr = static_cast<int64_t>(slot_of(k)) * p.sk_rows + r;
      const float w = ex2(p.part_lse[sr] * kLog2e - mb);
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + sr * D + col);
      wsum += w;
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const int tok = q0 + r / p.G, hq = g * p.G + r % p.G;
    float inv, lse;
    finish_row(M, wsum, p.sinks, hq, &inv, &lse);
    T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
             static_cast<int64_t>(hq) * p.o_sh + col;
    uint2 pk;
    pk.x = pack2<T>(acc.x * inv, acc.y * inv);
    pk.y = pack2<T>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
    if (p.lse && col == 0)
      p.lse[static_cast<int64_t>(hq) * p.total_q + tok] = lse;
  }
}

// Ring depth per configuration (two CTAs per SM).  D = 128, 16-bit: two
// stages of 32 KB (measured on GB300 against three: the same on the batched
// decode, 0.610 against 0.633-0.645 ms on 8 x 131072 keys); E4M3: three
// stages of 128 keys (32 KB); D = 64: six of 16 KB.
#ifndef PKV_DSK_D64_STAGES
#define PKV_DSK_D64_STAGES 6
#endif
#ifndef PKV_DSK_D128_STAGES
#define PKV_DSK_D128_STAGES 2
#endif
#ifndef PKV_DSK_D256_STAGES
#define PKV_DSK_D256_STAGES 2
#endif
#ifndef PKV_DSK_FP8_D128_KT
#define PKV_DSK_FP8_D128_KT 128
#endif
#ifndef PKV_DSK_FP8_D128_STAGES
#define PKV_DSK_FP8_D128_STAGES 3
#endif
#ifndef PKV_DSK_FP8_D256_STAGES
#define PKV_DSK_FP8_D256_STAGES 4
#endif

// Per instantiation: the shared-memory opt-in done on which devices, and
// the resident CTAs per SM found there.
template <typename T, int D, int NCW, int KT, int STAGES, bool KV8,
          bool Q8>
struct Inst {
  using C = Cfg<D, NCW, KT, STAGES, KV8, Q8>;
  static std::atomic<int> per_sm[kMaxDevices];

  static cudaError_t prepare(int dev, int* ctas_per_sm) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int n = per_sm[dev].load(std::memory_order_acquire);
    if (n <= 0) {
      auto kern = decode_sk_kernel<T, D, NCW, KT, STAGES, KV8, Q8>;
      cudaError_t e =
          smem_opt_in(reinterpret_cast<const void*>(kern), C::SMEM);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::NT,
                                                        C::SMEM);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      per_sm[dev].store(n, std::memory_order_release);
    }
    *ctas_per_sm = n;
    return cudaSuccess;
  }

  static cudaError_t launch(const AttnParams& p, const CUtensorMap& mk,
                            const CUtensorMap& mv, int grid, bool pdl,
                            cudaStream_t stream) {
    note_launch();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, decode_sk_kernel<T, D, NCW, KT, STAGES, KV8, Q8>, p, mk, mv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
};
template <typename T, int D, int NCW, int KT, int STAGES, bool KV8,
          bool Q8>
std::atomic<int> Inst<T, D, NCW, KT, STAGES, KV8, Q8>::per_sm[kMaxDevices];

// The configuration per (head size, cache type, query type); f(Inst) is
// called with the matching instantiation.
template <typename T, bool KV8, bool Q8, typename F>
cudaError_t with_cfg(int D, F&& f) {
  if constexpr (KV8) {
    switch (D) {
      case 128:
        return f(Inst<T, 128, 4, PKV_DSK_FP8_D128_KT, PKV_DSK_FP8_D128_STAGES,
                      true, Q8>{});
      case 256:
        return f(Inst<T, 256, 2, 32, PKV_DSK_FP8_D256_STAGES, true, Q8>{});
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (D) {
      case 64:
        return f(Inst<T, 64, 4, 64, PKV_DSK_D64_STAGES, false, false>{});
      case 128:
        return f(Inst<T, 128, 4, 64, PKV_DSK_D128_STAGES, false, false>{});
      case 256:
        return f(Inst<T, 256, 2, 32, PKV_DSK_D256_STAGES, false, false>{});
      default: return cudaErrorInvalidValue;
    }
  }
}

template <typename T, typename F>
cudaError_t dispatch_t(bool kv8, bool q8, int D, F&& f) {
  if (!kv8) return with_cfg<T, false, false>(D, f);
  return q8 ? with_cfg<T, true, true>(D, f) : with_cfg<T, true, false>(D, f);
}

template <typename F>
cudaError_t dispatch(bool bf16, bool kv8, bool q8, int D, F&& f) {
  if (q8 && !kv8) return cudaErrorInvalidValue;
  return bf16 ? dispatch_t<__nv_bfloat16>(kv8, q8, D, f)
              : dispatch_t<__half>(kv8, q8, D, f);
}

}  // namespace dsk

bool decode_sk_supported(int D, bool kv8) {
  return kv8 ? (D == 128 || D == 256) : (D == 64 || D == 128 || D == 256);
}

cudaError_t decode_sk_ctas(int D, bool bf16, bool kv8, bool q8, int sms,
                           int* ctas) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per = 0;
  e = dsk::dispatch(bf16, kv8, q8, D, [&](auto inst) {
    return decltype(inst)::prepare(dev, &per);
  });
  if (e != cudaSuccess) return e;
  *ctas = per * sms;
  return cudaSuccess;
}

namespace {

// Scratch layout of a launch with `ctas` CTAs (one chunk each) and partial
// slots of `rows` rows: two partial slots per chunk (O fp32 [rows][D] and
// LSE [rows]), then the chunk marks.
struct SkLayout {
  int chunks;
  size_t o_off, lse_off, marks_off, total;
};
size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
SkLayout sk_layout(int D, int ctas, int rows) {
  SkLayout l;
  l.chunks = ctas;
  const size_t slots = static_cast<size_t>(2) * l.chunks;
  l.o_off = 0;
  l.lse_off = a256(slots * rows * D * 4);
  l.marks_off = l.lse_off + a256(slots * rows * 4);
  l.total = l.marks_off + a256(static_cast<size_t>(l.chunks) * 8);
  return l;
}

}  // namespace

size_t decode_sk_workspace_bytes(int D, int ctas, int rows) {
  return sk_layout(D, ctas, rows).total;
}

cudaError_t launch_decode_attn_sk(const AttnParams& a, int D, bool bf16,
                                  int ctas, int rows, void* scratch,
                                  bool pdl, cudaStream_t stream) {
  AttnParams p = a;
  const bool kv8 = p.kv_fp8 != 0, q8 = p.q_fp8 != 0;
  const SkLayout l = sk_layout(D, ctas, rows);
  char* ws = static_cast<char*>(scratch);
  p.part_o = reinterpret_cast<float*>(ws + l.o_off);
  p.part_lse = reinterpret_cast<float*>(ws + l.lse_off);
  p.sk_marks = reinterpret_cast<int2*>(ws + l.marks_off);
  p.sk_chunks = l.chunks;
  p.sk_rows = rows;
  cudaError_t e = dsk::dispatch(bf16, kv8, q8, D, [&](auto inst) {
    using I = decltype(inst);
    const int KT = I::C::KTILE;
    int RB = 16;
    while (RB * 2 <= KT && p.BS % (RB * 2) == 0) RB *= 2;
    if (p.cu_k) RB = KT;    // non-paged: a box may start on any row
    p.rb = RB;
    p.kv_order_hnd = p.c_sh > p.c_sr ? 1 : 0;
    CUtensorMap mk, mv;
    const int elem = kv8 ? 0 : (bf16 ? 2 : 1);
    if (!make_kv_map_ex(&mk, p.kc, elem, D, p.BS, p.Hkv, p.num_blocks,
                        p.c_sb, p.c_sr, p.c_sh, RB, p.kv_order_hnd) ||
        !make_kv_map_ex(&mv, p.vc, elem, D, p.BS, p.Hkv, p.num_blocks,
                        p.c_sb, p.c_sr, p.c_sh, RB, p.kv_order_hnd))
      return cudaErrorInvalidValue;
    return I::launch(p, mk, mv, ctas, pdl, stream);
  });
  if (e != cudaSuccess || l.chunks < 2) return e;
  // the fold as a programmatic dependent launch: its blocks are resident
  // (waiting) when the decode grid ends, instead of launching after it
  note_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.chunks - 1));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int nch = l.chunks;
  switch (D) {
    case 64:
      e = bf16 ? cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__nv_bfloat16, 64>, p, nch)
               : cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__half, 64>, p, nch);
      break;
    case 128:
      e = bf16 ? cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__nv_bfloat16, 128>, p, nch)
               : cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__half, 128>, p, nch);
      break;
    default:
      e = bf16 ? cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__nv_bfloat16, 256>, p, nch)
               : cudaLaunchKernelEx(&cfg, dsk::fold_kernel<__half, 256>, p, nch);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
