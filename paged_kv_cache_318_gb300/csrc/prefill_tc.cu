// Prefill attention on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (flash_attn_varlen_func over the paged cache for requests with more
// than one query: cu_seqlens_q, seqused_k, block_table, causal, window_size,
// softcap, alibi_slopes, LSE) and cascade_attention (the shared prefix is one
// non-causal "sequence" of all the batch's queries).
//
// One CTA owns 128 packed query rows of one (request, KV head): packed row R
// is token R / G, query head g * G + R % G, so the G query heads of a KV head
// share every K/V tile.  The key range is walked in tiles of BN keys:
//
//   S_j  = Q K_j^T           tcgen05.mma kind::f16, M=128, N=BN, K=D, fp32 in
//                            TMEM (two S buffers, so S_{j+1} runs while the
//                            softmax warps work on S_j)
//   P_j  = exp2(S_j - m)     4 softmax warps, one thread per row (TMEM lane),
//                            written to shared memory as bf16/fp16
//   O   += P_j V_j           tcgen05.mma, M=128, N=D, K=BN, fp32 in TMEM
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue, warp 4 issues the
// MMAs (one elected lane) and owns the TMEM allocation, warp 5 issues TMA
// loads of K/V pages through the block table (one 2-D box of RB rows x 64
// elements per page and 64-column block, 128-byte swizzle) into a 2-stage
// ring.  Stages and S/P/O hand-offs are tracked with mbarriers; tcgen05.commit
// arrives on them when the MMAs finish.
//
// The running max is only moved when it grows by more than 2^8 (log2 units),
// so the O rescale (a TMEM load/multiply/store) is rare; softmax values then
// stay below 256, well inside bf16/fp32 range, and the final 1/l uses the
// same reference max, so the result is unchanged.
//
// Every mbarrier wait is bounded.  A wait that runs out sets the device error
// word (kErrTimeout), raises a CTA-wide abort flag, and every role drains its
// in-flight copies and MMAs before the TMEM is freed and the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>
#include <type_traits>

#include "pkv_common.cuh"
#include "tma_util.cuh"

namespace pkv {
namespace tc {

constexpr int BM = 128;
// The head-size-256 kernel: softmax warps 0-7, the MMA warp, the K and V
// loaders.
constexpr int NUM_THREADS = 352;
constexpr int MMA_WARP = 8;
constexpr int LOAD_WARP = 9;       // warps 9 (K) and 10 (V)
constexpr float kRescaleThreshold = 8.f;   // log2 units

// Tile geometry per head size.  D <= 128: 64-key tiles, one P buffer and
// 256 TMEM columns, so two CTAs share an SM (their prologues, epilogues and
// softmax phases overlap).  D = 256: 64-key tiles, two P buffers, all 512
// TMEM columns, one CTA per SM.
template <int D>
struct Cfg {
  static constexpr int BN = 64;   // keys per tile (one S row = 64 registers)
  static constexpr int NCB = D / 64;                 // 64-column blocks of D
  static constexpr int PCB = BN / 64;                // 64-column blocks of P
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;        // one K or V tile
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int STAGES = 2;
  static constexpr int PBUF = D <= 128 ? 1 : 2;      // P buffers
  static constexpr int S_COL = 0;                    // S buffers at 0, BN
  static constexpr int O_COL = 2 * BN;
  static constexpr int TMEM_NEED = 2 * BN + D;
  static constexpr int TMEM_COLS = TMEM_NEED <= 128 ? 128
                                   : (TMEM_NEED <= 256 ? 256 : 512);
  static_assert(TMEM_NEED <= TMEM_COLS, "TMEM budget");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + PBUF * P_BYTES;
  static constexpr int BAR_BYTES = 192;
  // the softmax warps' exchange of row maxima and sums between the two
  // key halves: [2 sets][2 halves][128 rows] floats
  static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;
  static constexpr int XCH_BYTES = 2 * 2 * 128 * 4;
  // The dynamic shared window starts 1024-byte aligned (checked at run
  // time); a CTA that takes all 512 TMEM columns also takes enough shared
  // memory that no second CTA fits beside it.
  static constexpr int SMEM_USED = OFF_XCH + XCH_BYTES;
  // no more CTAs per SM than TMEM can hold (512 columns per SM)
  static constexpr int SMEM_FLOOR = TMEM_COLS == 512 ? 120 * 1024
                                    : (TMEM_COLS == 256 ? 80 * 1024 : 0);
  static constexpr int SMEM = SMEM_USED < SMEM_FLOOR ? SMEM_FLOOR : SMEM_USED;
};

struct TcParams {
  const void* q;
  int64_t q_st, q_sh;
  void* out;
  int64_t o_st, o_sh;
  float* lse;
  int total_q;
  const int32_t* cu_q;
  const int32_t* seqused_k;
  const int32_t* cu_k;    // non-paged mode: rows cu_k[b] .. of one K/V tensor
  int total_k;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  int64_t num_blocks;
  int Hq, Hkv, G, BS, RB;
  float scale, softcap;
  const float* alibi;
  const float* sinks;
  const float* k_scale;   // fp8-sourced caches: value = code * scale
  const float* v_scale;
  int causal, wl, wr;
  int min_rows;
  int batch;
  int n_items;            // persistent kernel: work items (an upper bound)
  int out_v8;             // output rows 32-byte aligned: 256-bit stores
  int kv_order_hnd;   // tensor-map dim order: 1 = (D, BS, Hkv, NB)
  // head-size-256 kernel: the K / V maps are 5-D row-group maps (one box
  // per page lands as [8-row group][64-column block][8 rows][64 columns])
  int kv_rg;
  int* sched;             // persistent kernel: zeroed item counter, or null
  int q_tma;              // persistent kernel: Q tiles arrive as TMA boxes
  // persistent kernel: the O of a full 128-row tile leaves through a TMA
  // store from the ring stage of the item's last K (tile A) or V (tile B)
  int o_tma;
  // persistent kernel split-KV: every pair tile's key tiles cut into
  // n_split ranges, one work item each; partials to pre_o / pre_lse
  int n_split;
  float* pre_o;           // [n_split, total_q, Hq, D] fp32, rows O / l
  float* pre_lse;         // [n_split, Hq, total_q] fp32, natural log
  unsigned* err;
};

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 encoding).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo,
                                          uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;     // descriptor version
  d |= static_cast<uint64_t>(2) << 61;     // SWIZZLE_128B
  return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool bf16,
                                             bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a,
                                        uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

// Warp-collective forms: every lane of the warp executes them with the same
// (warp-uniform) operands and one lane, chosen by elect.sync, issues.  This
// keeps the descriptors in uniform registers.
__device__ __forceinline__ void mma_f16_warp(uint32_t d_tmem, uint64_t a,
                                             uint64_t b, uint32_t id,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster."
      "b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 columns of fp32 from TMEM.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
      "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
      "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])),
      "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
      "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// Packed pair arithmetic on the FMA pipe (one instruction for two fp32
// values): (a0, a1) = (a0, a1) * s + c and (s0, s1) += (a0, a1).
__device__ __forceinline__ void fma2(float& a0, float& a1, float s, float c) {
  uint64_t a, sv, cv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cv) : "f"(c));
  asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(a) : "l"(sv), "l"(cv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}
__device__ __forceinline__ void add2(float& s0, float& s1, float a0,
                                     float a1) {
  uint64_t sv, av;
  asm("mov.b64 %0, {%1, %2};" : "=l"(sv) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a0), "f"(a1));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(sv) : "l"(av));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(sv));
}

// max(a, b, c) in one instruction (three-input max, sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// min(max(a + b, 0), 1): the saturating add of the FMA pipe.
__device__ __forceinline__ float add_sat(float a, float b) {
  float d;
  asm("add.rn.sat.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// (s0, s1) <- (s0, s1) * m + c, one packed FMA.
__device__ __forceinline__ void fma2_pair(float& s0, float& s1, float m,
                                          float c) {
  uint64_t sv, mv, cv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(sv) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(mv) : "f"(m));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cv) : "f"(c));
  asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(sv) : "l"(mv), "l"(cv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(sv));
}

// ------------------------------------------------------------------ kernel

// Final logit (log2 units) of one score, with soft-cap, ALiBi and the
// admissibility mask of query position `pos` (general, per-element path).

__device__ __forceinline__ float masked_logit(float s, int key, int pos,
                                              bool valid, int kmin, int kmax,
                                              const TcParams& p, float slope,
                                              float qk_scale) {
  float x = s * qk_scale;
  if (p.softcap > 0.f) x = p.softcap * tanh_fast(x / p.softcap);
  if (p.alibi) x -= slope * fabsf(float(pos - key));
  x *= kLog2e;
  bool adm = valid && key >= kmin && key < kmax;
  if (p.causal) adm = adm && key <= pos;
  if (p.wl >= 0) adm = adm && key >= pos - p.wl;
  if (p.wr >= 0) adm = adm && key <= pos + p.wr;
  return adm ? x : -INFINITY;
}

template <typename T, int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
prefill_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  // a launch queued after this one as its programmatic dependent (the
  // cascade's suffix decode) may take the SMs this grid leaves free
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = Cfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t base_u = smem_u32(smem_raw);
  unsigned char* base = smem_raw;
  if (base_u & 1023u) {            // 128-byte swizzle atoms need 1 KB
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  // Compact grid: blockIdx.x = tile_index * Hkv + g, tiles of all
  // prefill-class requests in batch order, each request's last (longest)
  // row tile first.  Each warp scans 32 requests per step (one round trip
  // to the cu_seqlens_q cache lines per 32 requests).
  const int g = blockIdx.x % p.Hkv;
  const int t_lin = blockIdx.x / p.Hkv;
  int b = -1, tile = 0, q0 = 0, q_len = 0;
  {
    int acc = 0;
    for (int base_b = 0; base_b < p.batch && b < 0; base_b += 32) {
      const int bb = base_b + lane;
      int s0 = 0, ql = 0, nt = 0;
      if (bb < p.batch) {
        s0 = p.cu_q[bb];
        ql = min(p.cu_q[bb + 1] - s0, p.total_q - s0);
        const int rb = (s0 >= 0 && ql > 0) ? ql * G : 0;
        nt = rb >= p.min_rows ? (rb + BM - 1) / BM : 0;
      }
      int incl = nt;                         // inclusive prefix over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const bool hit = t_lin >= acc + incl - nt && t_lin < acc + incl;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int src = __ffs(m) - 1;
        b = base_b + src;
        const int excl = __shfl_sync(0xffffffffu, incl - nt, src);
        const int ntb = __shfl_sync(0xffffffffu, nt, src);
        q0 = __shfl_sync(0xffffffffu, s0, src);
        q_len = __shfl_sync(0xffffffffu, ql, src);
        tile = ntb - 1 - (t_lin - acc - excl);
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (b < 0) return;
  const int rows = q_len * G;
  const int row0 = tile * BM;
  const int row_end = min(rows, row0 + BM);
  const int koff = p.cu_k ? p.cu_k[b] : 0;     // non-paged: first key row
  const int L = p.cu_k ? p.cu_k[b + 1] - koff : p.seqused_k[b];
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  const int L_tab = p.cu_k ? (koff < 0 ? 0 : max(0, min(L, p.total_k - koff)))
                           : min(L, p.max_blocks * p.BS);
  if (L_tab < L && threadIdx.x == 0) atomicOr(p.err, kErrBadTable);
  int kmin, kmax;
  key_range(L, q_len, row0 / G, (row_end - 1) / G, p.causal, p.wl, p.wr, kmin,
            kmax);
  kmax = min(kmax, L_tab);
  const int RB = p.RB;
  const int kstart = (kmin / RB) * RB;
  const int n_tiles = kmax > kmin ? (kmax - kstart + BN - 1) / BN : 0;
  const int ctx = L - q_len;
  // Keys every valid row of this CTA admits: tiles inside [full_lo,
  // full_hi) need no per-element mask.
  const int p_lo = ctx + row0 / G, p_hi = ctx + (row_end - 1) / G;
  int full_lo = kmin, full_hi = kmax;
  if (p.wl >= 0) full_lo = max(full_lo, p_hi - p.wl);
  if (p.causal) full_hi = min(full_hi, p_lo + 1);
  if (p.wr >= 0) full_hi = min(full_hi, p_lo + p.wr + 1);
  const bool plain = p.softcap <= 0.f && p.alibi == nullptr;
  T* __restrict__ OUT = static_cast<T*>(p.out);

  if (n_tiles == 0) {
    // no admissible key for any row of the tile: out = 0, lse = -inf
    for (int i = tid; i < (row_end - row0) * (D / 8); i += NUM_THREADS) {
      const int r = row0 + i / (D / 8), c = i % (D / 8);
      const int tok = q0 + r / G, h = g * G + r % G;
      *reinterpret_cast<uint4*>(OUT + static_cast<int64_t>(tok) * p.o_st +
                                static_cast<int64_t>(h) * p.o_sh + c * 8) =
          make_uint4(0, 0, 0, 0);
      if (p.lse && c == 0)
        p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
            p.sinks ? p.sinks[h] : -INFINITY;
    }
    return;
  }

  const uint32_t sQ = base_u + C::OFF_Q;
  const uint32_t sK = base_u + C::OFF_K;
  const uint32_t sV = base_u + C::OFF_V;
  const uint32_t sP = base_u + C::OFF_P;
  const uint32_t bar0 = base_u + C::OFF_BAR;
  auto k_full = [&](int s) { return bar0 + 8 * (0 + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (4 + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (6 + s); };
  auto s_full = [&](int s) { return bar0 + 8 * (8 + s); };
  auto s_free = [&](int s) { return bar0 + 8 * (10 + s); };
  auto p_full = [&](int s) { return bar0 + 8 * (12 + s); };
  auto pv_done = [&](int s) { return bar0 + 8 * (14 + s); };
  const uint32_t final_bar = bar0 + 8 * 16;
  // x_bar(q): the two softmax warps of TMEM lane quarter q (one per key
  // half) have written their exchange value
  auto x_bar = [&](int q) { return bar0 + 8 * (19 + q); };
  static_assert(8 * 23 <= C::BAR_BYTES, "barrier area");
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(base + C::OFF_BAR + 8 * 18);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(base + C::OFF_BAR + 8 * 18 + 4);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 256);             // every softmax thread
      mbar_init(p_full(s), 256);
      mbar_init(pv_done(s), 1);
    }
    mbar_init(final_bar, 1);
    for (int q = 0; q < 4; ++q) mbar_init(x_bar(q), 64);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::
            "r"(smem_u32(tmem_slot)),
        "r"(C::TMEM_COLS)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"
                 ::: "memory");
  }

  // Q tile: packed rows, zero past row_end, 128-byte swizzled column blocks
  {
    const T* Q = static_cast<const T*>(p.q);
    for (int i = tid; i < BM * (D / 8); i += NUM_THREADS) {
      const int r = i / (D / 8), ch = i % (D / 8);
      const int R = row0 + r;
      const bool ok = R < row_end;
      const T* src = Q;
      if (ok)
        src = Q + static_cast<int64_t>(q0 + R / G) * p.q_st +
              static_cast<int64_t>(g * G + R % G) * p.q_sh + ch * 8;
      cp_async_16(sQ + (ch >> 3) * (BM * 128) + sw128(r, ch & 7), src,
                  ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // K / V tile layout in shared memory.  4-D boxes (RB rows of one 64-column
  // block each) give [column block][key][64]; the 5-D row-group boxes give
  // [8-key group][column block][8 keys][64].  Either way a 128-byte swizzle
  // atom is 8 keys x 64 columns: cbs is the stride between column blocks,
  // gs between 8-key groups.
  const uint32_t cbs = p.kv_rg ? 1024u : static_cast<uint32_t>(BN * 128);
  const uint32_t gs = p.kv_rg ? static_cast<uint32_t>(C::NCB * 1024) : 1024u;
  if (warp >= LOAD_WARP) {
    // --------------------------------------------------------- producers
    // Warp LOAD_WARP fills the K ring, the next warp the V ring, so a K
    // tile never waits behind a V stage.  Lane i issues the box of page i
    // of a tile and meanwhile fetches page i of the next tile, which keeps
    // block-table latency off the critical path.
    const int mat = warp - LOAD_WARP;
    const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    auto fetch = [&](int j) -> int {
      const int k0 = kstart + j * BN + lane * RB;
      if (j >= n_tiles || lane >= BN / RB || k0 >= kmax) return 0;
      if (p.cu_k) return 0;
      const int blk = __ldg(bt + k0 / p.BS);
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.err, kErrBadBlock);
        return 0;
      }
      return blk;
    };
    const void* tm = mat ? static_cast<const void*>(&tm_v)
                         : static_cast<const void*>(&tm_k);
    const uint32_t ring = mat ? sV : sK;
    int iss = 0;
    int cur = fetch(0);
    for (int j = 0; j < n_tiles; ++j) {
      const int nxt = fetch(j + 1);
      const int s = j & 1;
      const int kt = kstart + j * BN;
      int nbox = (kmax - kt + RB - 1) / RB;
      if (nbox > BN / RB) nbox = BN / RB;
      const uint32_t full = mat ? v_full(s) : k_full(s);
      int stop = 0;
      if (lane == 0) {
        const uint32_t empty = mat ? v_empty(s) : k_empty(s);
        if (j >= 2 &&
            !mbar_wait(empty, ((j >> 1) & 1) ^ 1, abort_flag, p.err))
          stop = 1;
        else
          mbar_expect_tx(full, nbox * C::NCB * RB * 128);
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (stop) break;
      if (lane < nbox) {
        const int k0 = kt + lane * RB;
        const int row = p.cu_k ? koff + k0 : k0 % p.BS;
        const uint32_t dst0 = ring + s * C::KV_BYTES;
        if (p.kv_rg) {
          // one box: RB / 8 key groups x every column block
          const uint32_t dst = dst0 + lane * (RB / 8) * gs;
          if (p.kv_order_hnd)
            tma_load_5d(dst, tm, 0, 0, 0, row >> 3, cur * p.Hkv + g, full);
          else
            tma_load_5d(dst, tm, 0, 0, 0, cur * (p.BS >> 3) + (row >> 3), g,
                        full);
        } else {
          for (int cb = 0; cb < C::NCB; ++cb) {
            const uint32_t dst = dst0 + cb * cbs + lane * RB * 128;
            if (p.kv_order_hnd)
              tma_load_4d(dst, tm, cb * 64, row, g, cur, full);
            else
              tma_load_4d(dst, tm, cb * 64, g, row, cur, full);
          }
        }
      }
      iss = j + 1;
      cur = nxt;
    }
    // drain: the last copies of each stage must land before the CTA exits
    if (lane == 0) {
      for (int t = max(0, iss - 2); t < iss; ++t)
        mbar_drain(mat ? v_full(t & 1) : k_full(t & 1), (t >> 1) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ---------------------------------------------------------- MMA issuer
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t ID_S = idesc(128, BN, kBF16, false);
    constexpr uint32_t ID_PV = idesc(128, D, kBF16, true);
    bool ok = true;
    auto do_pv = [&](int i) -> bool {
      const int s = i & 1;
      const int pb = i % C::PBUF;
      if (!mbar_wait(p_full(pb), (i / C::PBUF) & 1, abort_flag, p.err))
        return false;
      if (!mbar_wait(v_full(s), (i >> 1) & 1, abort_flag, p.err)) return false;
      // zero V rows that hold no key of this request (beyond seqused_k, or
      // pages that were not loaded), so 0 * garbage never reaches O
      const int kt = kstart + i * BN;
      int nbox = (kmax - kt + RB - 1) / RB;
      if (nbox > BN / RB) nbox = BN / RB;
      const int r0 = min(nbox * RB, max(L - kt, 0));
      if (r0 < BN) {
        const uint32_t v0 = sV + s * C::KV_BYTES;
        for (int idx = lane; idx < (BN - r0) * 8 * C::NCB; idx += 32) {
          const int cb = idx / ((BN - r0) * 8);
          const int rem = idx - cb * ((BN - r0) * 8);
          const int r = r0 + rem / 8, c = rem % 8;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                           v0 + (r >> 3) * gs + cb * cbs + (r & 7) * 128 +
                           (c << 4)),
                       "r"(0)
                       : "memory");
        }
        fence_proxy_async();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t v0 = sV + s * C::KV_BYTES;
        const uint32_t p0 = sP + pb * C::P_BYTES;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t a = sdesc(p0 + (k >> 2) * (BM * 128) + (k & 3) * 32,
                                   16, 1024);
          const uint64_t bdesc = sdesc(v0 + k * 2 * gs, cbs, gs);
          mma_f16(tmem + C::O_COL, a, bdesc, ID_PV, (i > 0 || k > 0) ? 1 : 0);
        }
        mma_commit(pv_done(pb));
        mma_commit(v_empty(s));
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int s = j & 1;
      if (!mbar_wait(k_full(s), (j >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      if (j >= 2 &&
          !mbar_wait(s_free(s), ((j - 2) >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t k0 = sK + s * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t a =
              sdesc(sQ + (k >> 2) * (BM * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t bdesc =
              sdesc(k0 + (k >> 2) * cbs + (k & 3) * 32, 16, gs);
          mma_f16(tmem + C::S_COL + s * BN, a, bdesc, ID_S, k > 0 ? 1 : 0);
        }
        mma_commit(s_full(s));
        mma_commit(k_empty(s));
      }
      __syncwarp();
      if (j >= 1 && !do_pv(j - 1)) ok = false;
    }
    if (ok) do_pv(n_tiles - 1);
    // all issued MMAs must finish before TMEM is released
    if (lane == 0) mma_commit(final_bar);
    __syncwarp();
    mbar_drain(final_bar, 0);
  } else {
    // ---------------------------------------------------- softmax warps
    // Eight warps: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its rows)
    // and the key half hf = w / 4 of each 64-key tile (and O columns
    // hf D / 2 ..), so two warps per SM sub-partition share each row's
    // softmax.  The halves agree on the row maximum (and, at the end, the
    // sum) through shared memory.
    const int hf = warp >> 2;                  // key half of every tile
    const int q4 = warp & 3;                   // TMEM lane quarter
    const int r = tid & 127;                   // row in tile == TMEM lane
    constexpr int BH = BN / 2;                 // keys of a half
    constexpr int DH = D / 2;                  // O columns of a half
    const int R = row0 + r;
    const bool valid = R < row_end;
    const int pos = ctx + (valid ? R / G : 0);
    const int h = g * G + (valid ? R % G : 0);
    const float slope = (p.alibi && valid) ? p.alibi[h] : 0.f;
    // caches converted from fp8: k_scale joins the logit scale, v_scale
    // multiplies the output
    const float qk_scale = p.scale * (p.k_scale ? *p.k_scale : 1.f);
    const float vscale = p.v_scale ? *p.v_scale : 1.f;
    const float scale_log2 = qk_scale * kLog2e;
    const float scale_over_cap = p.softcap > 0.f ? qk_scale / p.softcap : 0.f;
    const float cap_log2e = p.softcap * kLog2e;
    const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    float* xch = reinterpret_cast<float*>(base + C::OFF_XCH);
    int x_cnt = 0;                             // exchanges so far
    // this row's value against the other key half's, in slot set `set`;
    // false on abort.  A tile's maximum goes to set j & 1: that set is
    // rewritten two tiles later, after an S MMA the MMA warp issues only
    // once P_j (every thread's p_full arrival, made after its read) is in.
    // The final sum uses the set the last maximum did not.
    auto swap_half = [&](int set, float mine, float& other) -> bool {
      float* slot = xch + set * 256 + r;
      slot[hf * 128] = mine;
      mbar_arrive(x_bar(q4));
      if (!mbar_wait(x_bar(q4), x_cnt & 1, abort_flag, p.err)) return false;
      ++x_cnt;
      other = slot[(hf ^ 1) * 128];
      return true;
    };
    float m_ref = -INFINITY, l = 0.f;          // l: this half's sum
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(s_full(sb), (j >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kt = kstart + j * BN;
      const int kth = kt + hf * BH;            // this half's first key
      const bool unmasked = kt >= full_lo && kt + BN <= full_hi;
      const bool fast = plain && unmasked;
      // soft-cap without ALiBi on an unmasked tile: no per-key mask
      const bool fast_cap = !plain && p.alibi == nullptr && unmasked;
      const uint32_t s_addr = tmem + lane_base + C::S_COL + sb * BN + hf * BH;
      // this half of the S row (32 fp32) in one load; S is free right after
      float v[BH];
      tmem_ld32(s_addr, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free(sb));
      // logits in log2 units (the plain path folds the scale into exp2)
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      // plain scores stay raw in the max (scale > 0: max(scale s) =
      // scale max(s)); the scale joins the exponent's FMA
      const bool raw = fast && scale_log2 > 0.f;
      if (raw) {
#pragma unroll
        for (int e = 0; e < BH; e += 2)
          mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], v[e], v[e + 1]);
      } else if (fast) {
#pragma unroll
        for (int e = 0; e < BH; ++e)
          mx8[e & 7] = fmaxf(mx8[e & 7], v[e] * scale_log2);
      } else if (fast_cap) {
#pragma unroll
        for (int e = 0; e < BH; e += 2) {
          float x0 = v[e], x1 = v[e + 1];
          fma2(x0, x1, scale_over_cap, 0.f);
          x0 = tanh_fast(x0);
          x1 = tanh_fast(x1);
          fma2(x0, x1, cap_log2e, 0.f);
          v[e] = x0;
          v[e + 1] = x1;
          mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], x0, x1);
        }
      } else {
        // keys outside this row's admissible interval [a_lo, a_hi)
        // (causal, window, the CTA's key range) become -inf; one interval
        // test per key keeps the unrolled code short (a per-key predicate
        // chain fills the instruction cache)
        int a_lo = kmin, a_hi = kmax;
        if (p.causal) a_hi = min(a_hi, pos + 1);
        if (p.wl >= 0) a_lo = max(a_lo, pos - p.wl);
        if (p.wr >= 0) a_hi = min(a_hi, pos + p.wr + 1);
        if (!valid) a_hi = a_lo;
        const int lo_rel = a_lo - kth;
        const int n_rel = max(a_hi - a_lo, 0);
#pragma unroll
        for (int e = 0; e < BH; ++e) {
          float xs = v[e] * qk_scale;
          if (p.softcap > 0.f) xs = p.softcap * tanh_fast(xs * inv_cap);
          if (p.alibi) xs -= slope * fabsf(float(pos - (kth + e)));
          const bool in = static_cast<unsigned>(e - lo_rel) <
                          static_cast<unsigned>(n_rel);
          v[e] = in ? xs * kLog2e : -INFINITY;
          mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
        }
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      if (raw) mx *= scale_log2;
      // the row's maximum over both halves
      float mx_o;
      if (!swap_half(sb, mx, mx_o)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, mx_o);
      const bool grow = mx > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - mx);      // m_ref = -inf -> 0
        m_ref = mx;
        l *= alpha;
      }
      const float base_m = (m_ref == -INFINITY) ? 0.f : m_ref;
      // O holds PV_0..PV_{j-1}: rescale this half of it once PV_{j-1} is
      // done (both halves of a row take the same decision)
      if (j >= 1 && __any_sync(0xffffffffu, grow)) {
        const int pb = (j - 1) % C::PBUF;
        if (!mbar_wait(pv_done(pb), ((j - 1) / C::PBUF) & 1, abort_flag,
                       p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
          float ov[32];
          const uint32_t ta = tmem + lane_base + C::O_COL + hf * DH + c * 32;
          tmem_ld32(ta, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= alpha;
          tmem_st32(ta, ov);
        }
        tmem_wait_st();
      }
      // P = exp2(logit - m)
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
      const float sc = fast ? scale_log2 : 1.f;
#pragma unroll
      for (int e = 0; e < BH; e += 2) {
        float x0 = v[e], x1 = v[e + 1];
        fma2(x0, x1, sc, -base_m);
        x0 = ex2(x0);
        x1 = ex2(x1);
        v[e] = x0;
        v[e + 1] = x1;
        add2(sum8[2 * ((e >> 1) & 3)], sum8[2 * ((e >> 1) & 3) + 1], x0, x1);
      }
      // P buffer j % PBUF was last read by PV_{j-PBUF}
      const int pbj = j % C::PBUF;
      if (j >= C::PBUF &&
          !mbar_wait(pv_done(pbj), ((j - C::PBUF) / C::PBUF) & 1, abort_flag,
                     p.err)) {
        ok = false;
        break;
      }
      // this half of the P row -> shared memory (K-major, 128-byte swizzle)
      const uint32_t p_row = sP + pbj * C::P_BYTES;
#pragma unroll
      for (int qq = 0; qq < BH / 8; ++qq) {
        const int q = hf * (BH / 8) + qq;        // 16-byte chunk of the row
        const float* e = v + qq * 8;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                         p_row + (q >> 3) * (BM * 128) + sw128(r, q & 7)),
                     "r"(pack2<T>(e[0], e[1])), "r"(pack2<T>(e[2], e[3])),
                     "r"(pack2<T>(e[4], e[5])), "r"(pack2<T>(e[6], e[7]))
                     : "memory");
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
           ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tc_fence_before();
      fence_proxy_async();
      mbar_arrive(p_full(pbj));
    }
    const int lb = (n_tiles - 1) % C::PBUF;
    float l_o = 0.f;
    if (ok && mbar_wait(pv_done(lb), ((n_tiles - 1) / C::PBUF) & 1,
                        abort_flag, p.err) &&
        swap_half(n_tiles & 1, l, l_o)) {
      tc_fence_after();
      float inv, lse_v;
      finish_row(m_ref, l + l_o, p.sinks, h, &inv, &lse_v);
      inv *= vscale;
      const int tok = q0 + (valid ? R / G : 0);
      T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
               static_cast<int64_t>(h) * p.o_sh + hf * DH;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        float ov[32];
        tmem_ld32(tmem + lane_base + C::O_COL + hf * DH + c * 32, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 pk;
            pk.x = pack2<T>(ov[e] * inv, ov[e + 1] * inv);
            pk.y = pack2<T>(ov[e + 2] * inv, ov[e + 3] * inv);
            pk.z = pack2<T>(ov[e + 4] * inv, ov[e + 5] * inv);
            pk.w = pack2<T>(ov[e + 6] * inv, ov[e + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = pk;
          }
        }
      }
      if (valid && p.lse && hf == 0)
        p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
            lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile(
        "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
        "r"(C::TMEM_COLS)
        : "memory");
  }
  // launched as a programmatic dependent of the call's decode kernels:
  // this grid ends after them, so that later work sees both
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------ two-tile (ping-pong) kernel
//
// For D <= 128 one CTA owns 256 packed rows as two 128-row Q tiles, A and B,
// that share every K/V tile.  Each Q tile has its own softmax warpgroup
// (warps 0-3 for A, 4-7 for B), two S buffers in TMEM, two P buffers in
// shared memory and its own O accumulator in TMEM, so a warpgroup never
// waits on the MMA of the tile it just finished, and the tensor core always
// has the other tile's work queued.  Warp 8 issues the MMAs; warps 9 and 10
// issue the TMA loads of K and V tiles (one lane per page box).

constexpr int PP_THREADS = 352;
constexpr int PP_MMA_WARP = 8;
constexpr int PP_LOAD_WARP = 9;    // warps 9 (K) and 10 (V)
constexpr int PP_ROWS = 2 * BM;

template <int D>
struct PPCfg {
  static constexpr int BN = 64;
  static constexpr int NCB = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;          // one Q tile
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int STAGES = 2;
  static constexpr int O_COL = 4 * BN;                // S[x][buf] below
  static constexpr int TMEM_COLS = 512;
  static_assert(4 * BN + 2 * D <= TMEM_COLS, "TMEM budget");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;   // P[x][buf]
  static constexpr int OFF_BAR = OFF_P + 4 * P_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES;
};

template <typename T, int D>
__global__ void __launch_bounds__(PP_THREADS, 1)
prefill_pp_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  // a launch queued after this one as its programmatic dependent (the
  // cascade's suffix decode) may take the SMs this grid leaves free
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = PPCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t base_u = smem_u32(smem_raw);
  unsigned char* base = smem_raw;
  if (base_u & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;

  // ---- work item: (request, 256-row pair tile, KV head)
  const int g = blockIdx.x % p.Hkv;
  const int t_lin = blockIdx.x / p.Hkv;
  int b = -1, tile = 0, q0 = 0, q_len = 0;
  {
    int acc = 0;
    for (int base_b = 0; base_b < p.batch && b < 0; base_b += 32) {
      const int bb = base_b + lane;
      int s0 = 0, ql = 0, nt = 0;
      if (bb < p.batch) {
        s0 = p.cu_q[bb];
        ql = min(p.cu_q[bb + 1] - s0, p.total_q - s0);
        const int rb = (s0 >= 0 && ql > 0) ? ql * G : 0;
        nt = rb >= p.min_rows ? (rb + PP_ROWS - 1) / PP_ROWS : 0;
      }
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const bool hit = t_lin >= acc + incl - nt && t_lin < acc + incl;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int src = __ffs(m) - 1;
        b = base_b + src;
        const int excl = __shfl_sync(0xffffffffu, incl - nt, src);
        const int ntb = __shfl_sync(0xffffffffu, nt, src);
        q0 = __shfl_sync(0xffffffffu, s0, src);
        q_len = __shfl_sync(0xffffffffu, ql, src);
        tile = ntb - 1 - (t_lin - acc - excl);
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (b < 0) return;
  const int rows = q_len * G;
  const int koff = p.cu_k ? p.cu_k[b] : 0;     // non-paged: first key row
  const int L = p.cu_k ? p.cu_k[b + 1] - koff : p.seqused_k[b];
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  const int L_tab = p.cu_k ? (koff < 0 ? 0 : max(0, min(L, p.total_k - koff)))
                           : min(L, p.max_blocks * p.BS);
  if (L_tab < L && threadIdx.x == 0) atomicOr(p.err, kErrBadTable);
  const int ctx = L - q_len;
  const int RB = p.RB;
  // per Q tile x: rows [rx0, rx_end), keys [kmn[x], kmx[x])
  int rx0[2], rx_end[2], kmn[2], kmx[2];
  bool has[2];
  int kmin_u = 0x7fffffff, kmax_u = 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    rx0[x] = tile * PP_ROWS + x * BM;
    rx_end[x] = min(rows, rx0[x] + BM);
    has[x] = rx_end[x] > rx0[x];
    kmn[x] = 0;
    kmx[x] = 0;
    if (has[x]) {
      key_range(L, q_len, rx0[x] / G, (rx_end[x] - 1) / G, p.causal, p.wl,
                p.wr, kmn[x], kmx[x]);
      kmx[x] = min(kmx[x], L_tab);
      if (kmx[x] > kmn[x]) {
        kmin_u = min(kmin_u, kmn[x]);
        kmax_u = max(kmax_u, kmx[x]);
      }
    }
  }
  const int kstart = kmax_u > 0 ? (kmin_u / RB) * RB : 0;
  const int n_tiles = kmax_u > 0 ? (kmax_u - kstart + BN - 1) / BN : 0;
  // tile ranges [tlo[x], tlo[x] + nx[x]) of each Q tile in the union
  int tlo[2], nx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (has[x] && kmx[x] > kmn[x]) {
      tlo[x] = (kmn[x] - kstart) / BN;
      nx[x] = (kmx[x] - kstart + BN - 1) / BN - tlo[x];
    } else {
      tlo[x] = 0;
      nx[x] = 0;
    }
  }
  T* __restrict__ OUT = static_cast<T*>(p.out);
  const bool plain = p.softcap <= 0.f && p.alibi == nullptr;

  const uint32_t sQ = base_u + C::OFF_Q;
  const uint32_t sK = base_u + C::OFF_K;
  const uint32_t sV = base_u + C::OFF_V;
  const uint32_t sP = base_u + C::OFF_P;
  const uint32_t bar0 = base_u + C::OFF_BAR;
  auto k_full = [&](int s) { return bar0 + 8 * (0 + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (4 + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (6 + s); };
  auto s_full = [&](int x, int s) { return bar0 + 8 * (8 + 2 * x + s); };
  auto s_free = [&](int x, int s) { return bar0 + 8 * (12 + 2 * x + s); };
  auto p_full = [&](int x, int s) { return bar0 + 8 * (16 + 2 * x + s); };
  auto pv_done = [&](int x, int s) { return bar0 + 8 * (20 + 2 * x + s); };
  const uint32_t final_bar = bar0 + 8 * 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_BAR + 8 * 26);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(base + C::OFF_BAR + 8 * 26 + 4);

  if (n_tiles > 0) {
    if (tid == 0) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(k_full(s), 1);
        mbar_init(v_full(s), 1);
        mbar_init(k_empty(s), 1);
        mbar_init(v_empty(s), 1);
        for (int x = 0; x < 2; ++x) {
          mbar_init(s_full(x, s), 1);
          mbar_init(s_free(x, s), 128);
          mbar_init(p_full(x, s), 128);
          mbar_init(pv_done(x, s), 1);
        }
      }
      mbar_init(final_bar, 1);
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == PP_MMA_WARP) {
      asm volatile(
          "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], "
          "%1;" ::"r"(smem_u32(tmem_slot)),
          "r"(C::TMEM_COLS)
          : "memory");
      asm volatile(
          "tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
              : "memory");
    }
    // Q tiles A and B: packed rows, zero past each tile's end
    const T* Q = static_cast<const T*>(p.q);
    for (int i = tid; i < PP_ROWS * (D / 8); i += PP_THREADS) {
      const int rr = i / (D / 8), ch = i % (D / 8);
      const int x = rr / BM, r = rr % BM;
      const int R = rx0[x] + r;
      const bool ok = R < rx_end[x];
      const T* src = Q;
      if (ok)
        src = Q + static_cast<int64_t>(q0 + R / G) * p.q_st +
              static_cast<int64_t>(g * G + R % G) * p.q_sh + ch * 8;
      cp_async_16(sQ + x * C::Q_BYTES + (ch >> 3) * (BM * 128) +
                      sw128(r, ch & 7),
                  src, ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = n_tiles > 0 ? *tmem_slot : 0;

  if (warp == PP_LOAD_WARP || warp == PP_LOAD_WARP + 1) {
    if (n_tiles > 0) {
      // ------------------------------------------------------ producers
      // warp 9 loads K tiles, warp 10 V tiles, so a K tile never waits for
      // the release of a V stage; lane i issues box i of each tile and
      // prefetches its page id one tile ahead
      const int mat = warp - PP_LOAD_WARP;       // 0: K, 1: V
      const int32_t* bt =
          p.block_table + static_cast<int64_t>(b) * p.bt_stride;
      auto fetch = [&](int j) -> int {
        const int k0 = kstart + j * BN + lane * RB;
        if (j >= n_tiles || lane >= BN / RB || k0 >= kmax_u) return 0;
        if (p.cu_k) return 0;
      const int blk = __ldg(bt + k0 / p.BS);
        if (blk < 0 || blk >= p.num_blocks) {
          atomicOr(p.err, kErrBadBlock);
          return 0;
        }
        return blk;
      };
      const void* tm = mat ? static_cast<const void*>(&tm_v)
                           : static_cast<const void*>(&tm_k);
      int issued = 0;
      int cur = fetch(0);
      for (int j = 0; j < n_tiles; ++j) {
        const int nxt = fetch(j + 1);
        const int s = j & 1;
        const int kt = kstart + j * BN;
        int nbox = (kmax_u - kt + RB - 1) / RB;
        if (nbox > BN / RB) nbox = BN / RB;
        const uint32_t full = mat ? v_full(s) : k_full(s);
        int stop = 0;
        if (lane == 0) {
          const uint32_t empty = mat ? v_empty(s) : k_empty(s);
          if (j >= 2 && !mbar_wait(empty, ((j >> 1) & 1) ^ 1, abort_flag,
                                   p.err))
            stop = 1;
          else
            mbar_expect_tx(full, nbox * C::NCB * RB * 128);
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
        if (lane < nbox) {
          const uint32_t dst0 = (mat ? sV : sK) + s * C::KV_BYTES;
          const int k0 = kt + lane * RB;
          const int row = p.cu_k ? koff + k0 : k0 % p.BS;
          for (int cb = 0; cb < C::NCB; ++cb) {
            const uint32_t dst = dst0 + cb * (BN * 128) + lane * RB * 128;
            if (p.kv_order_hnd)
              tma_load_4d(dst, tm, cb * 64, row, g, cur, full);
            else
              tma_load_4d(dst, tm, cb * 64, g, row, cur, full);
          }
        }
        issued = j + 1;
        cur = nxt;
      }
      if (lane == 0) {
        for (int t = max(0, issued - 2); t < issued; ++t)
          mbar_drain(mat ? v_full(t & 1) : k_full(t & 1), (t >> 1) & 1);
      }
    }
  } else if (warp == PP_MMA_WARP) {
    if (n_tiles > 0) {
      // ---------------------------------------------------- MMA issuer
      constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
      constexpr uint32_t ID_S = idesc(128, BN, kBF16, false);
      constexpr uint32_t ID_PV = idesc(128, D, kBF16, true);
      bool ok = true;
      auto in_range = [&](int x, int j) {
        return j >= tlo[x] && j < tlo[x] + nx[x];
      };
      auto do_pv = [&](int i) -> bool {
        const int s = i & 1;
        if (!mbar_wait(v_full(s), (i >> 1) & 1, abort_flag, p.err))
          return false;
        const int kt = kstart + i * BN;
        int nbox = (kmax_u - kt + RB - 1) / RB;
        if (nbox > BN / RB) nbox = BN / RB;
        const int r0 = min(nbox * RB, max(L - kt, 0));
        if (r0 < BN) {
          const uint32_t v0 = sV + s * C::KV_BYTES;
          for (int idx = lane; idx < (BN - r0) * 8 * C::NCB; idx += 32) {
            const int cb = idx / ((BN - r0) * 8);
            const int rem = idx - cb * ((BN - r0) * 8);
            const int r = r0 + rem / 8, c = rem % 8;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             v0 + cb * (BN * 128) + r * 128 + (c << 4)),
                         "r"(0)
                         : "memory");
          }
          fence_proxy_async();
          __syncwarp();
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!in_range(x, i)) continue;
          const int ix = i - tlo[x];
          const int pb = ix & 1;
          if (!mbar_wait(p_full(x, pb), (ix >> 1) & 1, abort_flag, p.err))
            return false;
          tc_fence_after();
          {
            // descriptors advance by (bytes >> 4) in the start-address field
            const uint64_t a0 =
                sdesc(sP + (2 * x + pb) * C::P_BYTES, 16, 1024);
            const uint64_t b0 = sdesc(sV + s * C::KV_BYTES, BN * 128, 1024);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
              mma_f16_warp(tmem + C::O_COL + x * D,
                           a0 + (((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4),
                           b0 + ((k * 16 * 128) >> 4), ID_PV,
                           (ix > 0 || k > 0) ? 1 : 0);
            mma_commit_warp(pv_done(x, pb));
          }
        }
        mma_commit_warp(v_empty(s));
        return true;
      };
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        if (!mbar_wait(k_full(s), (j >> 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || !in_range(x, j)) continue;
          const int jx = j - tlo[x];
          const int sb = jx & 1;
          if (jx >= 2 && !mbar_wait(s_free(x, sb), ((jx - 2) >> 1) & 1,
                                    abort_flag, p.err)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          {
            const uint64_t a0 = sdesc(sQ + x * C::Q_BYTES, 16, 1024);
            const uint64_t b0 = sdesc(sK + s * C::KV_BYTES, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_f16_warp(tmem + (2 * x + sb) * BN,
                           a0 + (((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4),
                           b0 + (((k >> 2) * (BN * 128) + (k & 3) * 32) >> 4),
                           ID_S, k > 0 ? 1 : 0);
            mma_commit_warp(s_full(x, sb));
          }
        }
        if (!ok) break;
        mma_commit_warp(k_empty(s));
        if (j >= 1 && !do_pv(j - 1)) ok = false;
      }
      if (ok) do_pv(n_tiles - 1);
      mma_commit_warp(final_bar);
      mbar_drain(final_bar, 0);
    }
  } else {
    // ---------------------------------------------- softmax warpgroups
    const int x = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = tid & 127;                  // row in tile == TMEM lane
    // per-tile values by select (no runtime-indexed local arrays)
    const int my_rx0 = x ? rx0[1] : rx0[0];
    const int my_rx_end = x ? rx_end[1] : rx_end[0];
    const bool my_has = x ? has[1] : has[0];
    const int my_tlo = x ? tlo[1] : tlo[0];
    const int my_nx = x ? nx[1] : nx[0];
    const int R = my_rx0 + r;
    const bool valid = R < my_rx_end;
    const int pos = ctx + (valid ? R / G : 0);
    const int h = g * G + (valid ? R % G : 0);
    const int tok = q0 + (valid ? R / G : 0);
    const float slope = (p.alibi && valid) ? p.alibi[h] : 0.f;
    // caches converted from fp8: k_scale joins the logit scale, v_scale
    // multiplies the output
    const float qk_scale = p.scale * (p.k_scale ? *p.k_scale : 1.f);
    const float vscale = p.v_scale ? *p.v_scale : 1.f;
    const float scale_log2 = qk_scale * kLog2e;
    const float scale_over_cap = p.softcap > 0.f ? qk_scale / p.softcap : 0.f;
    const float cap_log2e = p.softcap * kLog2e;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int kmin = x ? kmn[1] : kmn[0], kmax = x ? kmx[1] : kmx[0];
    int full_lo = kmin, full_hi = kmax;
    if (my_has) {
      const int p_lo = ctx + my_rx0 / G, p_hi = ctx + (my_rx_end - 1) / G;
      if (p.wl >= 0) full_lo = max(full_lo, p_hi - p.wl);
      if (p.causal) full_hi = min(full_hi, p_lo + 1);
      if (p.wr >= 0) full_hi = min(full_hi, p_lo + p.wr + 1);
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int jx = 0; jx < my_nx; ++jx) {
      const int sb = jx & 1;
      if (!mbar_wait(s_full(x, sb), (jx >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kt = kstart + (my_tlo + jx) * BN;
      const bool unmasked = kt >= full_lo && kt + BN <= full_hi;
      const bool fast = plain && unmasked;
      const bool fast_cap = !plain && p.alibi == nullptr && unmasked;
      float v[BN];
      const uint32_t s_addr = tmem + lane_base + (2 * x + sb) * BN;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, v + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free(x, sb));
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      if (fast) {
#pragma unroll
        for (int e = 0; e < BN; ++e)
          mx8[e & 7] = fmaxf(mx8[e & 7], v[e] * scale_log2);
      } else if (fast_cap) {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          v[e] = cap_log2e * tanh_fast(v[e] * scale_over_cap);
          mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          v[e] = masked_logit(v[e], kt + e, pos, valid, kmin, kmax, p, slope,
                               qk_scale);
          mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
        }
      }
      const float mx =
          fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const bool grow = mx > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - mx);
        m_ref = mx;
        l *= alpha;
      }
      const float base_m = (m_ref == -INFINITY) ? 0.f : m_ref;
      if (jx >= 1 && __any_sync(0xffffffffu, grow)) {
        const int pb = (jx - 1) & 1;
        if (!mbar_wait(pv_done(x, pb), ((jx - 1) >> 1) & 1, abort_flag,
                       p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          const uint32_t ta = tmem + lane_base + C::O_COL + x * D + c * 32;
          tmem_ld32(ta, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= alpha;
          tmem_st32(ta, ov);
        }
        tmem_wait_st();
      }
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
      if (fast) {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          v[e] = ex2(fmaf(v[e], scale_log2, -base_m));
          sum8[e & 7] += v[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          v[e] = ex2(v[e] - base_m);
          sum8[e & 7] += v[e];
        }
      }
      // P buffer sb was last read by PV_x(jx - 2)
      if (jx >= 2 && !mbar_wait(pv_done(x, sb), ((jx - 2) >> 1) & 1,
                                abort_flag, p.err)) {
        ok = false;
        break;
      }
      const uint32_t p_row = sP + (2 * x + sb) * C::P_BYTES;
#pragma unroll
      for (int q = 0; q < BN / 8; ++q) {
        const float* e = v + q * 8;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                         p_row + (q >> 3) * (BM * 128) + sw128(r, q & 7)),
                     "r"(pack2<T>(e[0], e[1])), "r"(pack2<T>(e[2], e[3])),
                     "r"(pack2<T>(e[4], e[5])), "r"(pack2<T>(e[6], e[7]))
                     : "memory");
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
           ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tc_fence_before();
      fence_proxy_async();
      mbar_arrive(p_full(x, sb));
    }
    T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
             static_cast<int64_t>(h) * p.o_sh;
    if (my_nx == 0) {
      // no admissible key for this tile's rows: out = 0, lse = -inf
      if (valid) {
#pragma unroll
        for (int c = 0; c < D; c += 8)
          *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
        if (p.lse)
          p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
              p.sinks ? p.sinks[h] : -INFINITY;
      }
    } else if (ok) {
      const int lb = (my_nx - 1) & 1;
      if (mbar_wait(pv_done(x, lb), ((my_nx - 1) >> 1) & 1, abort_flag,
                    p.err)) {
        tc_fence_after();
        float inv, lse_v;
        finish_row(m_ref, l, p.sinks, h, &inv, &lse_v);
      inv *= vscale;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(tmem + lane_base + C::O_COL + x * D + c * 32, ov);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 pk;
              pk.x = pack2<T>(ov[e] * inv, ov[e + 1] * inv);
              pk.y = pack2<T>(ov[e + 2] * inv, ov[e + 3] * inv);
              pk.z = pack2<T>(ov[e + 4] * inv, ov[e + 5] * inv);
              pk.w = pack2<T>(ov[e + 6] * inv, ov[e + 7] * inv);
              *reinterpret_cast<uint4*>(dst + c * 32 + e) = pk;
            }
          }
        }
        if (valid && p.lse)
          p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
              lse_v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == PP_MMA_WARP && n_tiles > 0) {
    tc_fence_after();
    asm volatile(
        "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
        "r"(C::TMEM_COLS)
        : "memory");
  }
  // launched as a programmatic dependent of the call's decode kernels:
  // this grid ends after them, so that later work sees both
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------- two-tile kernel with P in tensor memory
//
// Same work split as prefill_pp_kernel (one CTA = two 128-row Q tiles of a
// (request, KV head), 8 softmax warps, one MMA warp, K and V loader warps),
// with 128-key tiles.  Tensor memory holds, per Q tile x, S_x (128 fp32
// columns) and O_x (D columns).  The softmax reads S_x into registers and
// writes P_x back as packed 16-bit pairs over the first 64 columns of S_x;
// the P V MMA then reads its A operand straight from tensor memory, so P
// never touches shared memory.  Because P_x overwrites S_x, the MMA warp
// issues P_x(j) V_j before S_x(j+1) = Q_x K_{j+1}^T (tcgen05 MMAs of one
// thread run in issue order); the overlap comes from the other Q tile,
// whose MMAs run while this tile's softmax works.
//
// Per key tile j of the union of both tiles' ranges the MMA warp issues
//   P_A(j-1) V_{j-1}, S_A(j), P_B(j-1) V_{j-1}, S_B(j)
// and each commit to s_full[x] also covers P_x(j-1) V_{j-1}, so when the
// softmax of tile x sees S_x(j) its O_x is complete (the rare rescale of
// O_x needs no extra wait).
constexpr int PT_THREADS = 384;
constexpr int PT_MMA_WARP = 8;
constexpr int PT_LOAD_WARP = 9;    // warps 9 (K) and 10 (V); warp 11: Q
// Work items (their geometry) travel through a ring of PT_ITEM_SLOTS
// shared-memory slots; every warp but warp 11 (which fills it) reads each
// slot once: 8 softmax warps, the MMA warp and the K and V loaders.
constexpr int PT_ITEM_SLOTS = 4;
constexpr int PT_ITEM_READERS = 11;
// Register split (setmaxnreg): the launch gives 168 per thread (384 x 168 =
// 64512); the softmax warpgroups take 200, warpgroup 2 keeps 96:
// 256 x 200 + 128 x 96 = 63488.  The launcher checks the 168.
constexpr int PT_LAUNCH_REGS = 168;
constexpr int PT_SOFTMAX_REGS = 200;
constexpr int PT_OTHER_REGS = 96;
static_assert(256 * PT_SOFTMAX_REGS + 128 * PT_OTHER_REGS <=
                  PT_THREADS * PT_LAUNCH_REGS,
              "register split exceeds the launch allocation");

template <int D>
struct PTCfg {
  static constexpr int BN = 128;
  static constexpr int NCB = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;          // one Q tile
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int STAGES = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int X_COLS = BN + D;               // S_x then O_x
  static_assert(2 * X_COLS <= TMEM_COLS, "TMEM budget");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int BAR_BYTES = 256;
  // ring of work items (PtItem, 112 bytes each) dealt by warp 11
  static constexpr int OFF_RING = OFF_BAR + BAR_BYTES;
  static constexpr int RING_BYTES = PT_ITEM_SLOTS * 112;
  // per-request metadata (cu_seqlens_q, key count, key offset) cached in
  // shared memory for batches up to META_MAX requests
  static constexpr int META_MAX = 2048;
  static constexpr int OFF_META = OFF_RING + RING_BYTES;
  static constexpr int META_BYTES = (3 * META_MAX + 4) * 4;
  static constexpr int SMEM = OFF_META + META_BYTES;
};

// 32 bytes to global memory in one store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* w) {
  asm volatile(
      "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
      "r"(w[6]), "r"(w[7])
      : "memory");
}

// D += A * B with A (M = 128 rows x K = 16, 16-bit) in tensor memory.
__device__ __forceinline__ void mma_f16_tmem_a_warp(uint32_t d_tmem,
                                                    uint32_t a_tmem,
                                                    uint64_t b, uint32_t id,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::
          "r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// Geometry of one work item (request b, 256-row pair tile, KV head g).
// pt_item computes it (a warp-wide scan over cu_seqlens_q; all lanes must
// call it; false for an index past the real items); the persistent kernel
// does that in one warp and hands the struct to the others through shared
// memory, so it is plain ints, 16-byte multiple in size.
struct PtItem {
  int item;                      // work-item index; -1 marks the end
  int b, g, q0, q_len, rows, L, ctx, koff, L_tab;
  int rx0[2], rx_end[2], kmn[2], kmx[2], tlo[2], nx[2];
  int has[2];
  int kstart, kmax_u, n_tiles;
  int split;                     // key split of a split-KV launch, else 0
};
static_assert(sizeof(PtItem) == 112, "PtItem is copied as 7 x 16 bytes");

struct PtMeta {
  const int* cu_q;     // [batch + 1]
  const int* len;      // [batch]: key count
  const int* koff;     // [batch]: first key row (non-paged), else 0
  bool cached;         // false: read the caller's arrays in global memory
};

// Items are (request, tile, KV head), each request's longest tiles first;
// with HM, (request, KV head, tile): tiles of one head consecutive.
template <bool HM>
__device__ __forceinline__ bool pt_item(const TcParams& p, int item, int lane,
                                        int BN, const PtMeta& md,
                                        PtItem& it) {
  const int G = p.G;
  it.g = HM ? 0 : item % p.Hkv;
  const int t_lin = HM ? item : item / p.Hkv;
  int b = -1, tile = 0, q0 = 0, q_len = 0;
  int acc = 0;
  for (int base_b = 0; base_b < p.batch && b < 0; base_b += 32) {
    const int bb = base_b + lane;
    int s0 = 0, ql = 0, nt = 0;
    if (bb < p.batch) {
      s0 = md.cached ? md.cu_q[bb] : p.cu_q[bb];
      const int s1 = md.cached ? md.cu_q[bb + 1] : p.cu_q[bb + 1];
      ql = min(s1 - s0, p.total_q - s0);
      const int rb = (s0 >= 0 && ql > 0) ? ql * G : 0;
      nt = rb >= p.min_rows ? (rb + PP_ROWS - 1) / PP_ROWS : 0;
      if constexpr (HM) nt *= p.Hkv;
    }
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const bool hit = t_lin >= acc + incl - nt && t_lin < acc + incl;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      const int src = __ffs(m) - 1;
      b = base_b + src;
      const int excl = __shfl_sync(0xffffffffu, incl - nt, src);
      const int ntb = __shfl_sync(0xffffffffu, nt, src);
      q0 = __shfl_sync(0xffffffffu, s0, src);
      q_len = __shfl_sync(0xffffffffu, ql, src);
      if constexpr (HM) {
        const int per = ntb / p.Hkv;          // tiles of one head
        const int j = t_lin - acc - excl;
        it.g = j / per;
        tile = per - 1 - (j - it.g * per);
      } else {
        tile = ntb - 1 - (t_lin - acc - excl);
      }
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (b < 0) return false;
  it.b = b;
  it.q0 = q0;
  it.q_len = q_len;
  it.rows = q_len * G;
  if (md.cached) {
    it.koff = md.koff[b];
    it.L = md.len[b];
  } else {
    it.koff = p.cu_k ? p.cu_k[b] : 0;        // non-paged: first key row
    it.L = p.cu_k ? p.cu_k[b + 1] - it.koff : p.seqused_k[b];
  }
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  it.L_tab = p.cu_k ? (it.koff < 0 ? 0 : max(0, min(it.L, p.total_k - it.koff)))
                    : min(it.L, p.max_blocks * p.BS);
  it.ctx = it.L - q_len;
  int kmin_u = 0x7fffffff, kmax_u = 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    it.rx0[x] = tile * PP_ROWS + x * BM;
    it.rx_end[x] = min(it.rows, it.rx0[x] + BM);
    it.has[x] = it.rx_end[x] > it.rx0[x];
    it.kmn[x] = 0;
    it.kmx[x] = 0;
    if (it.has[x]) {
      key_range(it.L, q_len, it.rx0[x] / G, (it.rx_end[x] - 1) / G, p.causal,
                p.wl, p.wr, it.kmn[x], it.kmx[x]);
      it.kmx[x] = min(it.kmx[x], it.L_tab);
      if (it.kmx[x] > it.kmn[x]) {
        kmin_u = min(kmin_u, it.kmn[x]);
        kmax_u = max(kmax_u, it.kmx[x]);
      }
    }
  }
  it.kmax_u = kmax_u;
  it.kstart = kmax_u > 0 ? (kmin_u / p.RB) * p.RB : 0;
  it.n_tiles = kmax_u > 0 ? (kmax_u - it.kstart + BN - 1) / BN : 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (it.has[x] && it.kmx[x] > it.kmn[x]) {
      it.tlo[x] = (it.kmn[x] - it.kstart) / BN;
      it.nx[x] = (it.kmx[x] - it.kstart + BN - 1) / BN - it.tlo[x];
    } else {
      it.tlo[x] = 0;
      it.nx[x] = 0;
    }
  }
  return true;
}

// Persistent: each CTA walks a sequence of work items; every role keeps
// running counters across items, so the loaders fetch the next item's K / V
// and warp 11 its Q while the softmax warps finish the previous item's
// output.  With p.sched (a zeroed counter) the items are dealt out at run
// time: a CTA starts with item blockIdx.x, and warp 11 claims the next one
// (gridDim.x + an atomic ticket) as the current one starts, so an SM that
// drew short items takes more of them and the SMs finish within about two
// items of each other.  Without a counter the items are blockIdx.x,
// blockIdx.x + gridDim.x, ...  Per item: q_full (Q in place),
// q_empty (the item's S MMAs are done with Q), o_ready (its MMAs are
// complete) and o_free[x] (the softmax of tile x has read O_x); the MMA
// warp waits o_free[x] of the previous item before it writes O_x again.
template <typename T, int D, bool HM = false>
__global__ void __launch_bounds__(PT_THREADS, 1)
prefill_ptmem_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_o) {
  // a launch queued after this one as its programmatic dependent (the
  // cascade's suffix decode) may take the SMs this grid leaves free
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = PTCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t base_u = smem_u32(smem_raw);
  unsigned char* base = smem_raw;
  if (base_u & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int RB = p.RB;

  const uint32_t sQ = base_u + C::OFF_Q;
  const uint32_t sK = base_u + C::OFF_K;
  const uint32_t sV = base_u + C::OFF_V;
  const uint32_t bar0 = base_u + C::OFF_BAR;
  auto k_full = [&](int s) { return bar0 + 8 * (0 + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (2 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (4 + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (6 + s); };
  auto s_full = [&](int x) { return bar0 + 8 * (8 + x); };
  auto p_full = [&](int x) { return bar0 + 8 * (10 + x); };
  auto o_free = [&](int x) { return bar0 + 8 * (12 + x); };
  // o_ready(x): every MMA of an item up to its last P_x V is complete
  auto o_ready = [&](int x) { return bar0 + 8 * (x ? 31 : 14); };
  const uint32_t q_full = bar0 + 8 * 15;
  const uint32_t q_empty = bar0 + 8 * 16;
  const uint32_t drain_bar = bar0 + 8 * 17;    // the MMA warp's final drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_BAR + 8 * 18);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(base + C::OFF_BAR + 8 * 18 + 4);
  // item ring: it_full[s] (warp 11 wrote slot s), it_empty[s] (all readers
  // are done with it)
  auto it_full = [&](int s) { return bar0 + 8 * (19 + s); };
  auto it_empty = [&](int s) { return bar0 + 8 * (19 + PT_ITEM_SLOTS + s); };
  static_assert(8 * (19 + 2 * PT_ITEM_SLOTS) <= C::BAR_BYTES, "barrier area");
  // per tile x and ring stage s: the tile's 128 threads have staged O in
  // stage s of K (x = 0) or V (x = 1); the K / V loader then stores it
  // with TMA and refills the stage
  auto stg_full = [&](int x, int st) { return bar0 + 8 * (27 + 2 * x + st); };
  static_assert(8 * 32 <= C::BAR_BYTES, "barrier area");
  static_assert(19 + 2 * PT_ITEM_SLOTS <= 27, "staging barriers overlap");
  const bool dyn = p.sched != nullptr;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(p_full(s), 128);
      mbar_init(o_free(s), 128);
    }
    mbar_init(o_ready(0), 1);
    mbar_init(o_ready(1), 1);
    for (int xx = 0; xx < 2; ++xx)
      for (int st = 0; st < 2; ++st) mbar_init(stg_full(xx, st), 128);
    mbar_init(q_full, p.q_tma ? 1 : 32);
    mbar_init(q_empty, 1);
    mbar_init(drain_bar, 1);
    for (int s = 0; s < PT_ITEM_SLOTS; ++s) {
      mbar_init(it_full(s), 1);
      mbar_init(it_empty(s), PT_ITEM_READERS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == PT_MMA_WARP) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], "
        "%1;" ::"r"(smem_u32(tmem_slot)),
        "r"(C::TMEM_COLS)
        : "memory");
    asm volatile(
        "tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
            : "memory");
  }
  // request metadata, read once per CTA instead of once per item and warp
  PtMeta md;
  {
    int* m_q = reinterpret_cast<int*>(base + C::OFF_META);
    int* m_len = m_q + C::META_MAX + 1;
    int* m_koff = m_len + C::META_MAX;
    md.cu_q = m_q;
    md.len = m_len;
    md.koff = m_koff;
    md.cached = p.batch <= C::META_MAX;
    if (md.cached) {
      for (int i = tid; i <= p.batch; i += PT_THREADS) {
        m_q[i] = p.cu_q[i];
        if (i < p.batch) {
          const int ko = p.cu_k ? p.cu_k[i] : 0;
          m_koff[i] = ko;
          m_len[i] = p.cu_k ? p.cu_k[i + 1] - ko : p.seqused_k[i];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = p.n_items;
  // The CTA's n-th item from the ring (all lanes of a reader warp call it,
  // in order n = 0, 1, ...): 1 = an item, 0 = no more items, -1 = abort.
  auto take_item = [&](int n, PtItem& it) -> int {
    const int s = n % PT_ITEM_SLOTS;
    if (!mbar_wait(it_full(s), (n / PT_ITEM_SLOTS) & 1, abort_flag, p.err))
      return -1;
    const int4* src =
        reinterpret_cast<const int4*>(base + C::OFF_RING + s * 112);
    int4 w[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) w[k] = src[k];
    memcpy(&it, w, sizeof(PtItem));
    __syncwarp();
    if (lane == 0) mbar_arrive(it_empty(s));
    return it.item >= 0 ? 1 : 0;
  };

  if (warp >= 8) {
  // warpgroup 2 (MMA, K / V loaders, Q loader) gives registers back to the
  // softmax warpgroups, all four warps on this one instruction
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PT_OTHER_REGS));
  if (warp == PT_LOAD_WARP || warp == PT_LOAD_WARP + 1) {
    // -------------------------------------------------------- K / V loaders
    // warp 9 loads K tiles, warp 10 V tiles; lane i issues box i of each
    // tile and prefetches its page id one tile ahead
    const int mat = warp - PT_LOAD_WARP;       // 0: K, 1: V
    const void* tm = mat ? static_cast<const void*>(&tm_v)
                         : static_cast<const void*>(&tm_k);
    int gj = 0;                                // tiles issued so far
    // O of this loader's tile (A for K, B for V) staged in ring stage st by
    // an epilogue and not yet stored: its box coordinates
    // (stage 0 and stage 1 kept apart, in registers)
    bool pend0 = false, pend1 = false;
    int g0 = 0, g1 = 0, tok0 = 0, tok1 = 0;
    int fl0 = 0, fl1 = 0;                      // stores done per stage
    // lane 0: store the O staged in stage st (after the 128 threads of the
    // tile have written it); false on abort
    auto flush = [&](int st) -> bool {
      if (!(st ? pend1 : pend0)) return true;
      const int fl = st ? fl1 : fl0;
      if (!mbar_wait(stg_full(mat, st), fl & 1, abort_flag, p.err))
        return false;
      if (st) { ++fl1; pend1 = false; } else { ++fl0; pend0 = false; }
      const uint32_t src = (mat ? sV : sK) + st * C::KV_BYTES;
      const int gg = st ? g1 : g0, tt = st ? tok1 : tok0;
#pragma unroll
      for (int cb = 0; cb < C::NCB; ++cb)
        tma_store_3d(&tm_o, src + cb * (BN * 128), cb * 64, gg * G, tt);
      bulk_commit();
      bulk_wait_read_all();
      return true;
    };
    bool ok = true;
    for (int n = 0; ok; ++n) {
      PtItem it;
      const int got = take_item(n, it);
      if (got <= 0) {
        ok = got == 0;
        break;
      }
      if (it.L_tab < it.L && lane == 0 && warp == PT_LOAD_WARP)
        atomicOr(p.err, kErrBadTable);
      const int32_t* bt =
          p.cu_k ? nullptr
                 : p.block_table + static_cast<int64_t>(it.b) * p.bt_stride;
      auto fetch = [&](int j) -> int {
        const int k0 = it.kstart + j * BN + lane * RB;
        if (j >= it.n_tiles || lane >= BN / RB || k0 >= it.kmax_u || !bt)
          return 0;
        const int blk = __ldg(bt + k0 / p.BS);
        if (blk < 0 || blk >= p.num_blocks) {
          atomicOr(p.err, kErrBadBlock);
          return 0;
        }
        return blk;
      };
      int cur = fetch(0);
      for (int j = 0; j < it.n_tiles; ++j, ++gj) {
        const int nxt = fetch(j + 1);
        const int s = gj & 1;
        const int kt = it.kstart + j * BN;
        int nbox = (it.kmax_u - kt + RB - 1) / RB;
        if (nbox > BN / RB) nbox = BN / RB;
        const uint32_t full = mat ? v_full(s) : k_full(s);
        int stop = 0;
        if (lane == 0) {
          const uint32_t empty = mat ? v_empty(s) : k_empty(s);
          if (gj >= 2 && !mbar_wait(empty, ((gj >> 1) & 1) ^ 1, abort_flag,
                                    p.err))
            stop = 1;
          // an epilogue staged O in this stage: store it before refilling
          else if (!flush(s))
            stop = 1;
          else
            mbar_expect_tx(full, nbox * C::NCB * RB * 128);
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) {
          ok = false;
          break;
        }
        if (lane < nbox) {
          const uint32_t dst0 = (mat ? sV : sK) + s * C::KV_BYTES;
          const int k0 = kt + lane * RB;
          const int row = p.cu_k ? it.koff + k0 : k0 % p.BS;
          for (int cb = 0; cb < C::NCB; ++cb) {
            const uint32_t dst = dst0 + cb * (BN * 128) + lane * RB * 128;
            if (p.kv_order_hnd)
              tma_load_4d(dst, tm, cb * 64, row, it.g, cur, full);
            else
              tma_load_4d(dst, tm, cb * 64, it.g, row, cur, full);
          }
        }
        cur = nxt;
      }
      // this item's tile staged by its epilogue in the stage of its last
      // K / V tile (the softmax warps use the same rule)
      if (p.o_tma && p.n_split <= 1 && it.nx[mat] > 0 &&
          it.rx_end[mat] - it.rx0[mat] == BM) {
        const int tt = it.q0 + it.rx0[mat] / G;
        if ((gj - 1) & 1) { pend1 = true; g1 = it.g; tok1 = tt; }
        else { pend0 = true; g0 = it.g; tok0 = tt; }
      }
    }
    if (lane == 0) {
      // the last items' staged O, then every store complete
      if (ok && (!flush(0) || !flush(1))) ok = false;
      bulk_wait_all();
      // no copy may be in flight when the CTA exits
      for (int t = max(0, gj - 2); t < gj; ++t)
        mbar_drain(mat ? v_full(t & 1) : k_full(t & 1), (t >> 1) & 1);
    }
  } else if (warp == PT_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Per item, rounds j = 1 .. n - 1 issue P_x(j - 1) V and S_x(j) for both
    // tiles.  The item's first S MMAs and its last P V MMAs go out at the
    // boundary with its neighbours: P_A(last) V, o_ready(A), the next
    // item's S_A(0), P_B(last) V, o_ready(B), S_B(0).  Each tile's epilogue
    // then starts when its own MMAs are done, while the other tile and the
    // next item keep the tensor pipe busy.
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t ID_S = idesc(128, BN, kBF16, false);
    constexpr uint32_t ID_PV = idesc(128, D, kBF16, true);
    bool ok = true;
    int gj = 0;                       // K / V tiles of earlier items
    int pv_cnt[2] = {0, 0};           // P_x V MMAs issued so far
    int n_done = 0;                   // items finished
    PtItem it;
    int got = take_item(0, it);
    ok = got >= 0;
    auto issue_s = [&](int x, int gk) {
      const uint64_t a0 = sdesc(sQ + x * C::Q_BYTES, 16, 1024);
      const uint64_t b0 = sdesc(sK + (gk & 1) * C::KV_BYTES, 16, 1024);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_f16_warp(tmem + x * C::X_COLS,
                     a0 + (((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4),
                     b0 + (((k >> 2) * (BN * 128) + (k & 3) * 32) >> 4),
                     ID_S, k > 0 ? 1 : 0);
      mma_commit_warp(s_full(x));
    };
    // the first round of item t (Q of item m, K / V tiles from gb): its S
    // MMAs, and q_empty when they are all of the item's; false on abort
    auto first_round = [&](const PtItem& t, int m, int gb) -> bool {
      if (!mbar_wait(q_full, m & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      bool k_here = false;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (t.n_tiles > 0 && t.tlo[x] == 0 && t.nx[x] > 0) {
          if (!k_here) {
            if (!mbar_wait(k_full(gb & 1), (gb >> 1) & 1, abort_flag, p.err))
              return false;
            tc_fence_after();
            k_here = true;
          }
          issue_s(x, gb);
        }
      }
      if (t.n_tiles > 0) mma_commit_warp(k_empty(gb & 1));
      if (t.n_tiles <= 1) mma_commit_warp(q_empty);
      return true;
    };
    if (got > 0 && !first_round(it, 0, 0)) ok = false;
    while (got > 0 && ok) {
      bool o_mine[2] = {n_done == 0, n_done == 0};   // O_x free to write
      auto claim_o = [&](int x) -> bool {
        if (o_mine[x]) return true;
        if (!mbar_wait(o_free(x), (n_done - 1) & 1, abort_flag, p.err))
          return false;
        tc_fence_after();
        o_mine[x] = true;
        return true;
      };
      auto in_range = [&](int x, int j) {
        return j >= it.tlo[x] && j < it.tlo[x] + it.nx[x];
      };
      // V_i resident (rows past the keys zeroed); false on abort
      auto v_ready = [&](int i) -> bool {
        const int gi = gj + i, s = gi & 1;
        if (!mbar_wait(v_full(s), (gi >> 1) & 1, abort_flag, p.err))
          return false;
        const int kt = it.kstart + i * BN;
        int nbox = (it.kmax_u - kt + RB - 1) / RB;
        if (nbox > BN / RB) nbox = BN / RB;
        const int r0 = min(nbox * RB, max(it.L - kt, 0));
        if (r0 < BN) {
          // rows past the last key may hold another request's NaN padding
          const uint32_t v0 = sV + s * C::KV_BYTES;
          for (int idx = lane; idx < (BN - r0) * 8 * C::NCB; idx += 32) {
            const int cb = idx / ((BN - r0) * 8);
            const int rem = idx - cb * ((BN - r0) * 8);
            const int r = r0 + rem / 8, c = rem % 8;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             v0 + cb * (BN * 128) + r * 128 + (c << 4)),
                         "r"(0)
                         : "memory");
          }
          fence_proxy_async();
          __syncwarp();
        }
        return true;
      };
      auto issue_pv = [&](int x, int i) -> bool {
        const int ix = i - it.tlo[x];
        if (ix == 0 && !claim_o(x)) return false;
        if (!mbar_wait(p_full(x), pv_cnt[x] & 1, abort_flag, p.err))
          return false;
        ++pv_cnt[x];
        tc_fence_after();
        const uint64_t b0 =
            sdesc(sV + ((gj + i) & 1) * C::KV_BYTES, BN * 128, 1024);
        const uint32_t s_col = tmem + x * C::X_COLS;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_f16_tmem_a_warp(s_col + BN, s_col + 8 * k,
                              b0 + ((k * 16 * 128) >> 4), ID_PV,
                              (ix > 0 || k > 0) ? 1 : 0);
        return true;
      };
      for (int j = 1; j < it.n_tiles && ok; ++j) {
        const int gk = gj + j;
        bool k_here = false;                 // K_j waited for
        if (!v_ready(j - 1)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (in_range(x, j - 1) && !issue_pv(x, j - 1)) {
            ok = false;
            break;
          }
          // V_{j-1} is free once both P V MMAs are done: release it before
          // S_B(j), so that the tile after next starts loading earlier
          if (x == 1) mma_commit_warp(v_empty((gk - 1) & 1));
          if (in_range(x, j)) {
            if (!k_here) {
              if (!mbar_wait(k_full(gk & 1), (gk >> 1) & 1, abort_flag,
                             p.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_here = true;
            }
            issue_s(x, gk);
          }
        }
        if (!ok) break;
        mma_commit_warp(k_empty(gk & 1));
        if (j == it.n_tiles - 1) mma_commit_warp(q_empty);
      }
      if (!ok) break;
      // ---- boundary: this item's last P V MMAs and o_ready per tile, the
      // next item's first S MMAs between them
      PtItem it_next;
      const int got_next = take_item(n_done + 1, it_next);
      if (got_next < 0) break;
      const int last = it.n_tiles - 1;
      const int gn = gj + it.n_tiles;        // the next item's first tile
      if (last >= 0 && !v_ready(last)) break;
      bool q_next = false, k_next = false;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (last >= 0 && in_range(x, last) && !issue_pv(x, last)) {
          ok = false;
          break;
        }
        // an item with no P_x V still waits for the epilogue before it, so
        // that no o_free phase is skipped
        if (!claim_o(x)) {
          ok = false;
          break;
        }
        mma_commit_warp(o_ready(x));
        if (x == 1 && last >= 0) mma_commit_warp(v_empty((gj + last) & 1));
        if (got_next > 0 && it_next.n_tiles > 0 && it_next.tlo[x] == 0 &&
            it_next.nx[x] > 0) {
          if (!q_next) {
            if (!mbar_wait(q_full, (n_done + 1) & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            q_next = true;
          }
          if (!k_next) {
            if (!mbar_wait(k_full(gn & 1), (gn >> 1) & 1, abort_flag,
                           p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            k_next = true;
          }
          issue_s(x, gn);
        }
      }
      if (!ok) break;
      if (got_next > 0) {
        // the rest of the next item's first round (as in first_round)
        if (!q_next) {
          if (!mbar_wait(q_full, (n_done + 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (it_next.n_tiles > 0) mma_commit_warp(k_empty(gn & 1));
        if (it_next.n_tiles <= 1) mma_commit_warp(q_empty);
      }
      gj += it.n_tiles;
      ++n_done;
      it = it_next;
      got = got_next;
    }
    // wait for every MMA of this CTA on a barrier no other role waits on (an
    // extra o_ready phase could complete before a softmax warp has waited
    // for the previous one, and the parity wait would then never return)
    mma_commit_warp(drain_bar);
    mbar_drain(drain_bar, 0);
  } else if (warp == PT_LOAD_WARP + 2) {
    // ------------------------------------ Q loader and item dealer (warp 11)
    // Slot n of the ring gets the CTA's n-th item (its PtItem; item = -1
    // ends every reader's loop).  Item n + 1 is chosen and published as
    // item n starts, so the loaders can fetch its first K / V tiles and the
    // MMA and softmax warps read its geometry while item n still runs.
    auto publish = [&](int n, const PtItem& it) -> bool {
      const int s = n % PT_ITEM_SLOTS;
      if (n >= PT_ITEM_SLOTS &&
          !mbar_wait(it_empty(s), ((n / PT_ITEM_SLOTS) - 1) & 1, abort_flag,
                     p.err))
        return false;
      if (lane == 0) {
        int4 w[7];
        memcpy(w, &it, sizeof(PtItem));
        int4* dst = reinterpret_cast<int4*>(base + C::OFF_RING + s * 112);
#pragma unroll
        for (int k = 0; k < 7; ++k) dst[k] = w[k];
        mbar_arrive(it_full(s));
      }
      return true;
    };
    int item = static_cast<int>(blockIdx.x);     // gridDim.x <= n_items
    int q_issued = 0;                            // Q loads as TMA boxes
    for (int n = 0;; ++n) {
      PtItem it;
      const int pair = p.n_split > 1 ? item / p.n_split : item;
      const bool real = item >= 0 && pt_item<HM>(p, pair, lane, BN, md, it);
      it.item = real ? item : -1;
      it.split = 0;
      if (real && p.n_split > 1) {
        // split s: key tiles [j0, j1) of the pair's union range; each Q
        // tile keeps its own range clipped to them
        const int s = item - pair * p.n_split;
        const int per = (it.n_tiles + p.n_split - 1) / p.n_split;
        const int j0 = min(s * per, it.n_tiles);
        const int j1 = min(j0 + per, it.n_tiles);
        const int k0 = it.kstart + j0 * BN, k1 = it.kstart + j1 * BN;
#pragma unroll
        for (int xs = 0; xs < 2; ++xs) {
          const int lo = max(it.tlo[xs], j0);
          const int hi = min(it.tlo[xs] + it.nx[xs], j1);
          if (hi > lo) {
            it.tlo[xs] = lo - j0;
            it.nx[xs] = hi - lo;
            it.kmn[xs] = max(it.kmn[xs], k0);
            it.kmx[xs] = min(it.kmx[xs], k1);
          } else {
            it.tlo[xs] = 0;
            it.nx[xs] = 0;
          }
        }
        it.kstart = k0;
        it.kmax_u = min(it.kmax_u, k1);
        it.n_tiles = j1 - j0;
        it.split = s;
      }
      if (!publish(n, it) || !real) break;
      // the previous item's S MMAs are done with Q
      if (n >= 1 && !mbar_wait(q_empty, (n - 1) & 1, abort_flag, p.err))
        break;
      if (p.q_tma) {
        // one box per (tile, 64 columns): 128 / G tokens x the G heads of
        // KV head g, which is the tile's 128 packed rows in order.  Rows
        // past the request are the next tokens' (or, past the tensor,
        // zeros): they only feed S rows no output is taken from.
        if (lane == 0) {
          mbar_expect_tx(q_full, (it.has[1] ? 2 : 1) * C::Q_BYTES);
#pragma unroll
          for (int xq = 0; xq < 2; ++xq) {
            if (!it.has[xq]) continue;
#pragma unroll
            for (int cb = 0; cb < C::NCB; ++cb)
              tma_load_3d(sQ + xq * C::Q_BYTES + cb * (BM * 128), &tm_q,
                          cb * 64, it.g * G, it.q0 + it.rx0[xq] / G, q_full);
          }
        }
        ++q_issued;
      } else {
        // both Q tiles: packed rows, zero past each tile's end; lane i
        // copies rows i, i + 32, ... (one address computation per row)
        const T* Q = static_cast<const T*>(p.q);
        for (int rr = lane; rr < PP_ROWS; rr += 32) {
          const int xq = rr / BM, rq = rr % BM;
          const int Rq = it.rx0[xq] + rq;
          const bool okq = Rq < it.rx_end[xq];
          const T* src = Q;
          if (okq)
            src = Q + static_cast<int64_t>(it.q0 + Rq / G) * p.q_st +
                  static_cast<int64_t>(it.g * G + Rq % G) * p.q_sh;
          const uint32_t dst = sQ + xq * C::Q_BYTES;
#pragma unroll
          for (int ch = 0; ch < D / 8; ++ch)
            cp_async_16(dst + (ch >> 3) * (BM * 128) + sw128(rq, ch & 7),
                        okq ? src + ch * 8 : src, okq ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();
        mbar_arrive(q_full);
      }
      // the next item: dealt at run time (an atomic ticket) or the fixed
      // stride; an index past the real items becomes the end marker
      if (dyn) {
        int v = 0;
        if (lane == 0)
          v = static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
        item = __shfl_sync(0xffffffffu, v, 0);
      } else {
        const int64_t i = blockIdx.x + static_cast<int64_t>(n + 1) * gridDim.x;
        item = i < n_items ? static_cast<int>(i) : -1;
      }
      if (item >= n_items) item = -1;
    }
    // no Q box may be in flight when the CTA exits (the MMA warp waits for
    // every one it uses, but not after an abort)
    if (lane == 0 && q_issued > 0) mbar_drain(q_full, (q_issued - 1) & 1);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PT_SOFTMAX_REGS));
    // ---------------------------------------------- softmax warpgroups
    const int x = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = tid & 127;                  // row in tile == TMEM lane
    T* __restrict__ OUT = static_cast<T*>(p.out);
    const bool plain = p.softcap <= 0.f && p.alibi == nullptr;
    const float qk_scale = p.scale * (p.k_scale ? *p.k_scale : 1.f);
    const float vscale = p.v_scale ? *p.v_scale : 1.f;
    const float scale_log2 = qk_scale * kLog2e;
    const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + x * C::X_COLS;
    const uint32_t o_addr = s_addr + BN;
    int s_cnt = 0;                            // S_x tiles seen so far
    int n_done = 0;
    int g_base = 0;                           // K / V tiles of earlier items
    bool ok = true;
    PtItem it;
    int got = take_item(0, it);
    ok = got >= 0;
    // this thread's row of tile x in an item: computed for the next item
    // while this one waits for its last MMAs (the code runs once per item
    // and would otherwise sit between the epilogue and the next softmax)
    struct RowGeo {
      int rx0, rx_end, tlo, nx, pos, h, tok, kmin, kmax, full_lo, full_hi;
      float slope;
      bool valid;
    };
    auto row_geo = [&](const PtItem& t) {
      RowGeo e;
      e.rx0 = x ? t.rx0[1] : t.rx0[0];
      e.rx_end = x ? t.rx_end[1] : t.rx_end[0];
      const bool has = x ? t.has[1] : t.has[0];
      e.tlo = x ? t.tlo[1] : t.tlo[0];
      e.nx = x ? t.nx[1] : t.nx[0];
      const int R = e.rx0 + r;
      e.valid = R < e.rx_end;
      e.pos = t.ctx + (e.valid ? R / G : 0);
      e.h = t.g * G + (e.valid ? R % G : 0);
      e.tok = t.q0 + (e.valid ? R / G : 0);
      e.slope = (p.alibi && e.valid) ? p.alibi[e.h] : 0.f;
      e.kmin = x ? t.kmn[1] : t.kmn[0];
      e.kmax = x ? t.kmx[1] : t.kmx[0];
      e.full_lo = e.kmin;
      e.full_hi = e.kmax;
      if (has) {
        const int p_lo = t.ctx + e.rx0 / G;
        const int p_hi = t.ctx + (e.rx_end - 1) / G;
        if (p.wl >= 0) e.full_lo = max(e.full_lo, p_hi - p.wl);
        if (p.causal) e.full_hi = min(e.full_hi, p_lo + 1);
        if (p.wr >= 0) e.full_hi = min(e.full_hi, p_lo + p.wr + 1);
      }
      return e;
    };
    RowGeo cg{};
    if (got > 0) cg = row_geo(it);
    while (got > 0 && ok) {
      const int my_rx0 = cg.rx0;
      const int my_rx_end = cg.rx_end;
      const int my_tlo = cg.tlo;
      const int my_nx = cg.nx;
      const bool valid = cg.valid;
      const int pos = cg.pos;
      const int h = cg.h;
      const int tok = cg.tok;
      const float slope = cg.slope;
      const int kmin = cg.kmin;
      const int kmax = cg.kmax;
      const int full_lo = cg.full_lo, full_hi = cg.full_hi;
      float m_ref = -INFINITY, l = 0.f;
      for (int jx = 0; jx < my_nx; ++jx, ++s_cnt) {
        if (!mbar_wait(s_full(x), s_cnt & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kt = it.kstart + (my_tlo + jx) * BN;
        const bool unmasked = kt >= full_lo && kt + BN <= full_hi;
        float v[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(s_addr + c * 32, v + c * 32);
        tmem_wait_ld();
        // logits in log2 units; keys outside this row's admissible
        // interval [a_lo, a_hi) (causal, window, item range) become -inf.
        // The interval test keeps the masked code short: a fully unrolled
        // per-key predicate chain over 128 keys overflows the instruction
        // cache.
        int lo_rel = 0, n_rel = BN;             // admissible e in [lo, lo+n)
        if (!unmasked) {
          int a_lo = kmin, a_hi = kmax;
          if (p.causal) a_hi = min(a_hi, pos + 1);
          if (p.wl >= 0) a_lo = max(a_lo, pos - p.wl);
          if (p.wr >= 0) a_hi = min(a_hi, pos + p.wr + 1);
          if (!valid) a_hi = a_lo;
          lo_rel = a_lo - kt;
          n_rel = max(a_hi - a_lo, 0);
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
        // plain scores stay raw: max(scale * s) = scale * max(s) for scale
        // > 0, and the scale joins the exponent's FMA
        const bool raw = plain && scale_log2 > 0.f;
        if (raw && unmasked) {
#pragma unroll
          for (int e = 0; e < BN; e += 2)
            mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], v[e], v[e + 1]);
        } else if (raw) {
          // a key outside [lo_rel, lo_rel + n_rel) becomes min(s, -2^126):
          // its flag f (1 out, 0 in) comes from saturating adds on the FMA
          // pipe and the bound 2^126 - f * 2^127 from one packed FMA, in
          // place of integer compares and a select per key on the ALU pipe.
          // The min also replaces a NaN score (a key row past the
          // request's end may hold one).
          constexpr float kBig = 8.50705917e37f;       // 2^126
          const int hi_rel = lo_rel + n_rel;
          if (p.wl < 0) {
            // no left window: lo_rel <= 0, only keys >= hi_rel are out;
            // f = sat(e + 1 - hi_rel)
            const float one_m_hi = static_cast<float>(1 - hi_rel);
#pragma unroll
            for (int e = 0; e < BN; e += 2) {
              float b0 = add_sat(static_cast<float>(e), one_m_hi);
              float b1 = add_sat(static_cast<float>(e + 1), one_m_hi);
              fma2_pair(b0, b1, -2.f * kBig, kBig);
              v[e] = fminf(v[e], b0);
              v[e + 1] = fminf(v[e + 1], b1);
              mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], v[e], v[e + 1]);
            }
          } else {
            // out iff |2e - (lo + hi - 1)| > hi - 1 - lo, i.e. f =
            // sat(|2e - c2| - r2) (the left side moves in steps of 2)
            const float c2 = static_cast<float>(lo_rel + hi_rel - 1);
            const float r2 = static_cast<float>(hi_rel - 1 - lo_rel);
#pragma unroll
            for (int e = 0; e < BN; e += 2) {
              float b0 = add_sat(fabsf(static_cast<float>(2 * e) - c2), -r2);
              float b1 =
                  add_sat(fabsf(static_cast<float>(2 * e + 2) - c2), -r2);
              fma2_pair(b0, b1, -2.f * kBig, kBig);
              v[e] = fminf(v[e], b0);
              v[e + 1] = fminf(v[e + 1], b1);
              mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], v[e], v[e + 1]);
            }
          }
        } else if (plain) {
#pragma unroll
          for (int e = 0; e < BN; ++e) {
            const bool in = static_cast<unsigned>(e - lo_rel) <
                            static_cast<unsigned>(n_rel);
            v[e] = in ? v[e] * scale_log2 : -INFINITY;
            mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
          }
        } else {
          // soft-cap and / or ALiBi (their own slower path)
#pragma unroll
          for (int e = 0; e < BN; ++e) {
            float xs = v[e] * qk_scale;
            if (p.softcap > 0.f) xs = p.softcap * tanh_fast(xs * inv_cap);
            if (p.alibi) xs -= slope * fabsf(float(pos - (kt + e)));
            const bool in = static_cast<unsigned>(e - lo_rel) <
                            static_cast<unsigned>(n_rel);
            v[e] = in ? xs * kLog2e : -INFINITY;
            mx8[e & 7] = fmaxf(mx8[e & 7], v[e]);
          }
        }
        float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]),
                         max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        // a row with every key of the tile out keeps -inf (its scores sit
        // at -2^126)
        if (raw) mx = mx < -0.5f * 8.50705917e37f ? -INFINITY : mx * scale_log2;
        const bool grow = mx > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2(m_ref - mx);
          m_ref = mx;
          l *= alpha;
        }
        const float base_m = (m_ref == -INFINITY) ? 0.f : m_ref;
        if (jx >= 1 && __any_sync(0xffffffffu, grow)) {
          // O_x is complete: the commit behind s_full covered P(j-1) V
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(o_addr + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
            tmem_st32(o_addr + c * 32, ov);
          }
        }
        float sum8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
        const float sc = raw ? scale_log2 : 1.f;
#pragma unroll
        for (int e = 0; e < BN; e += 2) {
          float x0 = v[e], x1 = v[e + 1];
          fma2(x0, x1, sc, -base_m);
          x0 = ex2(x0);
          x1 = ex2(x1);
          v[e] = x0;
          v[e + 1] = x1;
          add2(sum8[2 * ((e >> 1) & 3)], sum8[2 * ((e >> 1) & 3) + 1], x0,
               x1);
        }
        // P_x over the first BN / 2 columns of S_x: column c holds the keys
        // 2c (low half) and 2c + 1 (high half)
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          float pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            pk[e] = __uint_as_float(pack2<T>(v[c * 64 + 2 * e],
                                             v[c * 64 + 2 * e + 1]));
          tmem_st32(s_addr + c * 32, pk);
        }
        l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
             ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(x));
      }
      if (!ok) break;
      // the next item's geometry, read before this item's output stores
      // (they hold up shared-memory access while they drain)
      PtItem it_next;
      const int got_next = take_item(n_done + 1, it_next);
      if (got_next < 0) break;
      RowGeo ng{};
      if (got_next > 0) ng = row_geo(it_next);
      // ---- epilogue: every MMA of the item is complete
      if (!mbar_wait(o_ready(x), n_done & 1, abort_flag, p.err)) break;
      tc_fence_after();

      T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
               static_cast<int64_t>(h) * p.o_sh;
      if (p.n_split > 1) {
        // split-KV partial of this row: O / l in fp32 and its LSE (the sink
        // joins once, in the combine); no key in the split: 0 and -inf
        float* po = p.pre_o + ((static_cast<int64_t>(it.split) * p.total_q +
                                tok) * p.Hq + h) * D;
        float* pl = p.pre_lse +
                    (static_cast<int64_t>(it.split) * p.Hq + h) * p.total_q +
                    tok;
        if (my_nx == 0) {
          tc_fence_before();
          mbar_arrive(o_free(x));
          if (valid) {
            const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < D; e += 8) st_global_v8(po + e, z);
            *pl = -INFINITY;
          }
        } else {
          float inv, lse_v;
          finish_row(m_ref, l, nullptr, h, &inv, &lse_v);
          inv *= vscale;
          float ov[D];
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            tmem_ld32(o_addr + c * 32, ov + c * 32);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(o_free(x));
          if (valid) {
#pragma unroll
            for (int e = 0; e < D; e += 8) {
              uint32_t w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q)
                w[q] = __float_as_uint(ov[e + q] * inv);
              st_global_v8(po + e, w);
            }
            *pl = lse_v;
          }
        }
      } else if (my_nx == 0) {
        // no admissible key for this tile's rows: out = 0, lse = -inf
        tc_fence_before();
        mbar_arrive(o_free(x));
        if (valid) {
#pragma unroll
          for (int c = 0; c < D; c += 8)
            *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
          if (p.lse)
            p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
                p.sinks ? p.sinks[h] : -INFINITY;
        }
      } else if (p.o_tma && my_rx_end - my_rx0 == BM) {
        // a full tile: O goes through the (consumed) ring stage of the
        // item's last K (tile A) or V (tile B) tile; that loader stores it
        // with one TMA store per 64 columns before it refills the stage
        float inv, lse_v;
        finish_row(m_ref, l, p.sinks, h, &inv, &lse_v);
        inv *= vscale;
        float ov[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tmem_ld32(o_addr + c * 32, ov + c * 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(o_free(x));              // O_x may be overwritten now
        const uint32_t stg = (x ? sV : sK) +
                             ((g_base + it.n_tiles - 1) & 1) * C::KV_BYTES;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t w0 = pack2<T>(ov[8 * c] * inv, ov[8 * c + 1] * inv);
          const uint32_t w1 =
              pack2<T>(ov[8 * c + 2] * inv, ov[8 * c + 3] * inv);
          const uint32_t w2 =
              pack2<T>(ov[8 * c + 4] * inv, ov[8 * c + 5] * inv);
          const uint32_t w3 =
              pack2<T>(ov[8 * c + 6] * inv, ov[8 * c + 7] * inv);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                           stg + (c >> 3) * (BN * 128) + sw128(r, c & 7)),
                       "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
        // the K / V loader stores the staged tile and then refills the stage
        fence_proxy_async();
        mbar_arrive(stg_full(x, (g_base + it.n_tiles - 1) & 1));
        if (p.lse) p.lse[static_cast<int64_t>(h) * p.total_q + tok] = lse_v;
      } else {
        float inv, lse_v;
        finish_row(m_ref, l, p.sinks, h, &inv, &lse_v);
        inv *= vscale;
        float ov[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tmem_ld32(o_addr + c * 32, ov + c * 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(o_free(x));              // O_x may be overwritten now
        if (valid) {
          if (p.out_v8) {
            // whole 32-byte sectors: half the store transactions of 16 B
#pragma unroll
            for (int e = 0; e < D; e += 16) {
              uint32_t w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q)
                w[q] = pack2<T>(ov[e + 2 * q] * inv, ov[e + 2 * q + 1] * inv);
              st_global_v8(dst + e, w);
            }
          } else {
#pragma unroll
            for (int e = 0; e < D; e += 8) {
              uint4 pk;
              pk.x = pack2<T>(ov[e] * inv, ov[e + 1] * inv);
              pk.y = pack2<T>(ov[e + 2] * inv, ov[e + 3] * inv);
              pk.z = pack2<T>(ov[e + 4] * inv, ov[e + 5] * inv);
              pk.w = pack2<T>(ov[e + 6] * inv, ov[e + 7] * inv);
              *reinterpret_cast<uint4*>(dst + e) = pk;
            }
          }
          if (p.lse) p.lse[static_cast<int64_t>(h) * p.total_q + tok] = lse_v;
        }
      }
      ++n_done;
      g_base += it.n_tiles;
      it = it_next;
      cg = ng;
      got = got_next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == PT_MMA_WARP) {
    tc_fence_after();
    asm volatile(
        "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
        "r"(C::TMEM_COLS)
        : "memory");
  }
  // launched as a programmatic dependent of the call's decode kernels:
  // this grid ends after them, so that later work sees both
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Fold the split-KV partials of prefill-class requests.  One warp per
// (token, query head) row, its lanes across D (D <= 128, S <= 16): M = the
// largest partial LSE (and the sink logit), w_s = e^(lse_s - M), out =
// sum w_s o_s / sum w_s, lse = M + ln sum w_s.  Every partial of the row is
// loaded before any is used, so the row costs one memory round trip.
// Grid: (rows / 8, 1, request).
constexpr int kPreMaxSplits = 16;
template <typename T>
__global__ void __launch_bounds__(256)
prefill_split_combine_kernel(const CombineParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int q0 = p.cu_q[b];
  const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
  if (q0 < 0 || q_len <= 0 || q_len * p.G < p.min_rows) return;
  const int row = blockIdx.x * 8 + warp;
  if (row >= q_len * p.Hq) return;
  const int tok = q0 + row / p.Hq, h = row - (row / p.Hq) * p.Hq;
  const int S = p.splits, D = p.D;
  const int c = lane * 4;
  float l[kPreMaxSplits];
  float4 v[kPreMaxSplits];
#pragma unroll
  for (int s = 0; s < kPreMaxSplits; ++s) {
    l[s] = -INFINITY;
    v[s] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s < S) {
      l[s] = p.part_lse[(static_cast<int64_t>(s) * p.Hq + h) * p.total_q +
                        tok];
      if (c < D)
        v[s] = *reinterpret_cast<const float4*>(
            p.part_o +
            ((static_cast<int64_t>(s) * p.total_q + tok) * p.Hq + h) * D + c);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kPreMaxSplits; ++s) M = fmaxf(M, l[s]);
  const float sink = p.sinks ? p.sinks[h] : -INFINITY;
  M = fmaxf(M, sink);
  const float base = (M == -INFINITY) ? 0.f : M;
  float lsum = p.sinks ? __expf(sink - base) : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kPreMaxSplits; ++s) {
    const float w = (l[s] == -INFINITY) ? 0.f : __expf(l[s] - base);
    lsum += w;
    acc.x += w * v[s].x;
    acc.y += w * v[s].y;
    acc.z += w * v[s].z;
    acc.w += w * v[s].w;
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  if (c < D) {
    T* dst = static_cast<T*>(p.out) + static_cast<int64_t>(tok) * p.o_st +
             static_cast<int64_t>(h) * p.o_sh + c;
    uint2 pk;
    pk.x = pack2<T>(acc.x * inv, acc.y * inv);
    pk.y = pack2<T>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  }
  if (p.lse && lane == 0)
    p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
        lsum > 0.f ? base + __logf(lsum) : -INFINITY;
}

// ------------------------------------------------------------ host side

}  // namespace tc

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 4-D map over one cache view: (D, Hkv, BS, NB) for NHD strides, (D, BS, Hkv,
// NB) when the head stride is the larger (HND); box = BOXC x 1 x RB x 1 with
// BOXC * element bytes = 128.
bool make_kv_map_ex(CUtensorMap* map, const void* ptr, int elem, int D,
                    int BS, int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                    int64_t s_head, int RB, bool hnd) {
  auto fn = encode_fn();
  if (!fn || elem < 0 || elem > 2) return false;
  const int eb = elem == 0 ? 1 : 2;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  dims[0] = D;
  dims[3] = static_cast<cuuint64_t>(NB);
  strides[2] = static_cast<cuuint64_t>(s_blk) * eb;
  box[0] = 128 / eb;
  box[3] = 1;
  if (hnd) {
    dims[1] = BS;  strides[0] = static_cast<cuuint64_t>(s_row) * eb;  box[1] = RB;
    dims[2] = Hkv; strides[1] = static_cast<cuuint64_t>(s_head) * eb; box[2] = 1;
  } else {
    dims[1] = Hkv; strides[0] = static_cast<cuuint64_t>(s_head) * eb; box[1] = 1;
    dims[2] = BS;  strides[1] = static_cast<cuuint64_t>(s_row) * eb;  box[2] = RB;
  }
  const CUtensorMapDataType dt =
      elem == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                : (elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  // L2 promotion: a 16-bit head row (D = 128: 256 bytes) arrives as two
  // 128-byte boxes of the same tile, so 256-byte lines waste nothing; a
  // one-byte-code row is 128 bytes, and 256-byte lines would also fetch the
  // next KV head's row, which another CTA reads at another time (measured:
  // 28 % more DRAM bytes than the codes on the fp8 batched decode)
  const CUtensorMapL2promotion promo =
      eb == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
              : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUresult r = fn(map, dt, 4, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D row-group map of a 16-bit cache view: (64 columns, 8 rows, D / 64
// column blocks, key groups, heads).  The key-group and the page axes merge
// into one when their strides line up, so one box of RB keys (RB / 8
// groups) covers every column block of one page and lands in shared memory
// as [8-key group][column block][8 keys][64 columns]: the NHD view needs
// s_blk = BS s_row (dims: groups of all pages, then heads), the HND view
// s_blk = Hkv s_head (dims: groups of a page, then page x head).  False when
// the view does not fit; the caller keeps the 4-D boxes then.
bool make_kv_rg_map(CUtensorMap* map, const void* ptr, bool bf16, int D,
                    int BS, int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                    int64_t s_head, int RB, bool hnd) {
  auto fn = encode_fn();
  if (!fn || D % 64 != 0 || BS % 8 != 0 || RB % 8 != 0 || RB > BS ||
      RB / 8 > 256)
    return false;
  const int64_t eb = 2;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(D / 64),
                       static_cast<cuuint32_t>(RB / 8), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  dims[0] = 64;
  dims[1] = 8;
  dims[2] = static_cast<cuuint64_t>(D / 64);
  strides[0] = static_cast<cuuint64_t>(s_row * eb);
  strides[1] = 128;
  strides[2] = static_cast<cuuint64_t>(8 * s_row * eb);
  strides[3] = static_cast<cuuint64_t>(s_head * eb);
  if (!hnd) {
    const int64_t groups = NB * (BS / 8);
    if (s_blk != BS * s_row || groups > 0x7fffffff) return false;
    dims[3] = static_cast<cuuint64_t>(groups);
    dims[4] = static_cast<cuuint64_t>(Hkv);
  } else {
    const int64_t ph = NB * Hkv;
    if (s_blk != Hkv * s_head || ph > 0x7fffffff) return false;
    dims[3] = static_cast<cuuint64_t>(BS / 8);
    dims[4] = static_cast<cuuint64_t>(ph);
  }
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  5, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_kv_map(CUtensorMap* map, const void* ptr, bool bf16, int D, int BS,
                 int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                 int64_t s_head, int RB, bool hnd) {
  return make_kv_map_ex(map, ptr, bf16 ? 2 : 1, D, BS, Hkv, NB, s_blk, s_row,
                        s_head, RB, hnd);
}


// 3-D map over the query rows [T, Hq, D] (element strides s_tok, s_head;
// unit stride along D): dims (D, Hq, T), box 64 x G x (128 / G), 128-byte
// swizzled.  One box holds 64 columns of the 128 packed rows (token, head of
// one KV group) of a Q tile, in the order and layout the S MMA reads.
// False when G does not divide 128 or the driver rejects the map.
static bool make_rows_map(CUtensorMap* map, const void* ptr, bool bf16, int D,
                          int Hq, int T, int64_t s_tok, int64_t s_head,
                          int G) {
  auto fn = encode_fn();
  if (!fn || G <= 0 || 128 % G != 0 || T <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s_head) * 2,
                           static_cast<cuuint64_t>(s_tok) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G),
                       static_cast<cuuint32_t>(128 / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map,
                  bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int prefill_tc_block_keys(int) { return 64; }

cudaError_t launch_prefill_split_combine(const CombineParams& p,
                                         int max_seqlen_q, bool bf16,
                                         cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(max_seqlen_q) * p.Hq;
  if (p.batch <= 0 || rows <= 0) return cudaSuccess;
  if ((rows + 7) / 8 > 0x7fffffff || p.batch > 65535 || p.D > 128 ||
      p.splits > tc::kPreMaxSplits)
    return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>((rows + 7) / 8), 1,
            static_cast<unsigned>(p.batch));
  note_launch();
  if (bf16)
    tc::prefill_split_combine_kernel<__nv_bfloat16>
        <<<grid, 256, 0, stream>>>(p);
  else
    tc::prefill_split_combine_kernel<__half><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_attn_tc(const AttnParams& a, int D, bool bf16,
                                   int grid_y, bool p_in_tmem,
                                   int* splits_used, cudaStream_t stream,
                                   bool pdl) {
  using namespace tc;
  if (splits_used) *splits_used = 1;
  TcParams p{};
  p.q = a.q;
  p.q_st = a.q_st;
  p.q_sh = a.q_sh;
  p.out = a.out;
  p.o_st = a.o_st;
  p.o_sh = a.o_sh;
  p.lse = a.lse;
  p.total_q = a.total_q;
  p.cu_q = a.cu_q;
  p.seqused_k = a.seqused_k;
  p.cu_k = a.cu_k;
  p.total_k = a.total_k;
  p.block_table = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.BS = a.BS;
  p.scale = a.scale;
  p.softcap = a.softcap;
  p.alibi = a.alibi;
  p.sinks = a.sinks;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.causal = a.causal;
  p.wl = a.wl;
  p.wr = a.wr;
  p.min_rows = a.min_rows;
  p.batch = a.batch;
  p.err = a.err;
  const int BN = prefill_tc_block_keys(D);
  int RB = 16;
  while (RB * 2 <= BN && a.BS % (RB * 2) == 0) RB *= 2;
  if (a.cu_k) RB = BN;    // non-paged: boxes may start on any row
  p.RB = RB;
  p.kv_order_hnd = a.c_sh > a.c_sr ? 1 : 0;
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) % 32 == 0 &&
              (a.o_st * 2) % 32 == 0 && (a.o_sh * 2) % 32 == 0)
                 ? 1
                 : 0;
  CUtensorMap mk, mv;
  // head size 256: one row-group box per page (4-D boxes cost one TMA
  // instruction per 64-column block, and the instruction rate, not the
  // bytes, bounded the loads)
  p.kv_rg = 0;
  if (D == 256 && !a.cu_k &&
      make_kv_rg_map(&mk, a.kc, bf16, D, a.BS, a.Hkv, a.num_blocks, a.c_sb,
                     a.c_sr, a.c_sh, RB, p.kv_order_hnd) &&
      make_kv_rg_map(&mv, a.vc, bf16, D, a.BS, a.Hkv, a.num_blocks, a.c_sb,
                     a.c_sr, a.c_sh, RB, p.kv_order_hnd))
    p.kv_rg = 1;
  else if (!make_kv_map(&mk, a.kc, bf16, D, a.BS, a.Hkv, a.num_blocks, a.c_sb,
                        a.c_sr, a.c_sh, RB, p.kv_order_hnd) ||
           !make_kv_map(&mv, a.vc, bf16, D, a.BS, a.Hkv, a.num_blocks, a.c_sb,
                        a.c_sr, a.c_sh, RB, p.kv_order_hnd))
    return cudaErrorInvalidValue;
  // compact 1-D grid: an upper bound on the row tiles of all requests,
  // sum_b ceil(q_b * G / rows) <= ceil(total_q * G / rows) + batch, with
  // 256-row pair tiles for D <= 128 and 128-row tiles for D = 256
  (void)grid_y;
  const bool pp = D <= 128;
  const int cta_rows = pp ? PP_ROWS : BM;
  const int64_t tiles =
      (static_cast<int64_t>(a.total_q) * a.G + cta_rows - 1) / cta_rows +
      a.batch;
  const int64_t gx = tiles * a.Hkv;
  if (gx <= 0 || gx > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(gx));
  p.n_items = static_cast<int>(gx);
  p.n_split = 1;
  // the launch configuration (programmatic dependent when pdl)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  auto config = [&](int threads, int smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
  };
  auto go = [&](void (*kern)(TcParams, CUtensorMap, CUtensorMap), int smem,
                int threads) -> cudaError_t {
    cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    note_launch();
    const cudaLaunchConfig_t cfg = config(threads, smem);
    e = cudaLaunchKernelEx(&cfg, kern, p, mk, mv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  };
  if (p_in_tmem) {
    // the register split inside the kernel assumes exactly PT_LAUNCH_REGS
    // per thread at launch; anything else falls back to the kernel that
    // stages P through shared memory
    static int regs[2][2] = {};
    const int bi = bf16 ? 1 : 0, di = D == 64 ? 0 : 1;
    if (D <= 128 && regs[bi][di] == 0) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(
          &fa, bf16 ? (D == 64 ? (const void*)prefill_ptmem_kernel<__nv_bfloat16, 64>
                               : (const void*)prefill_ptmem_kernel<__nv_bfloat16, 128>)
                    : (D == 64 ? (const void*)prefill_ptmem_kernel<__half, 64>
                               : (const void*)prefill_ptmem_kernel<__half, 128>));
      if (e != cudaSuccess) return e;
      regs[bi][di] = fa.numRegs;
    }
    if (D <= 128 && regs[bi][di] != PT_LAUNCH_REGS) p_in_tmem = false;
  }
  if (p_in_tmem && D <= 128) {
    // persistent: one CTA per SM walks the items (an item needs two 128-row
    // Q tiles of packed rows, so the item count is that of the pair grid)
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess || sms <= 0)
      sms = 1;
    // split-KV: each pair tile's keys in a.pre_splits ranges, one item
    // each, when the caller planned it (few items for the SMs)
    int64_t items = gx;
    if (a.pre_splits > 1 && a.pre_o && a.pre_lse &&
        gx * a.pre_splits <= 0x7fffffff) {
      p.n_split = a.pre_splits;
      p.pre_o = a.pre_o;
      p.pre_lse = a.pre_lse;
      items = gx * a.pre_splits;
      p.n_items = static_cast<int>(items);
      if (splits_used) *splits_used = a.pre_splits;
    }
    grid = dim3(static_cast<unsigned>(items));
    if (a.max_ctas > 0 && a.max_ctas < sms) sms = a.max_ctas;
    if (static_cast<int64_t>(sms) < items) {
      grid = dim3(static_cast<unsigned>(sms));
      // items dealt at run time when the caller's workspace holds a
      // counter, unless there are many per SM: those are small (the bound
      // counts a tile per request), and a ticket's round trip before each
      // one then costs more than the balance gains (measured: 700 requests
      // of 1-200 tokens, about 39 items per SM, ran 10 % faster in the
      // fixed order; 9.7 per SM ran 2 % faster dealt at run time)
      if (a.sched && items <= 16 * static_cast<int64_t>(sms)) {
        if (!a.sched_zeroed) {
          cudaError_t e = cudaMemsetAsync(a.sched, 0, sizeof(int), stream);
          if (e != cudaSuccess) return e;
        }
        p.sched = a.sched;
      }
    }
  }
  if (p_in_tmem && D <= 128) {
    // Q tiles as TMA boxes when the KV group size divides the 128-row tile
    // (the rows of a tile are then whole tokens); else cp.async rows
    CUtensorMap mq;
    memset(&mq, 0, sizeof(mq));
    p.q_tma = make_rows_map(&mq, a.q, bf16, D, a.Hq, a.total_q, a.q_st,
                            a.q_sh, a.G)
                  ? 1
                  : 0;
    // the output map has the same box (a tile's 128 packed rows, 64
    // columns); unsplit launches only (split partials are fp32 rows)
    CUtensorMap mo;
    memset(&mo, 0, sizeof(mo));
    p.o_tma = (p.q_tma && p.n_split == 1 &&
               make_rows_map(&mo, a.out, bf16, D, a.Hq, a.total_q, a.o_st,
                             a.o_sh, a.G))
                  ? 1
                  : 0;
    auto go3 = [&](void (*kern)(TcParams, CUtensorMap, CUtensorMap,
                                CUtensorMap, CUtensorMap),
                   int smem) -> cudaError_t {
      cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), smem);
      if (e != cudaSuccess) return e;
      note_launch();
      const cudaLaunchConfig_t cfg = config(PT_THREADS, smem);
      e = cudaLaunchKernelEx(&cfg, kern, p, mk, mv, mq, mo);
      if (e != cudaSuccess) return e;
      return cudaGetLastError();
    };
    // one item per CTA (D = 128): the order only places the items on the
    // SMs, and head by head the CTAs that share a head's K/V sit together
    // (the cascade's prefix: 0.1331 -> 0.1289 ms); with more items than
    // CTAs, longest-first across heads wins (varlen prefill 0.2310 against
    // 0.2700 ms head by head).  A separate instantiation: the extra branch
    // in the item scan slowed the usual kernel by 1.5 %.
    const bool hm = D == 128 && static_cast<int64_t>(grid.x) >= p.n_items;
    if (hm) {
      static int hm_regs[2] = {};
      auto hk = bf16 ? (const void*)prefill_ptmem_kernel<__nv_bfloat16, 128, true>
                     : (const void*)prefill_ptmem_kernel<__half, 128, true>;
      int& r = hm_regs[bf16 ? 1 : 0];
      if (r == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, hk);
        if (e != cudaSuccess) return e;
        r = fa.numRegs;
      }
      if (r == PT_LAUNCH_REGS)
        return bf16 ? go3(prefill_ptmem_kernel<__nv_bfloat16, 128, true>,
                          PTCfg<128>::SMEM)
                    : go3(prefill_ptmem_kernel<__half, 128, true>,
                          PTCfg<128>::SMEM);
    }
    if (bf16)
      return D == 64 ? go3(prefill_ptmem_kernel<__nv_bfloat16, 64>,
                           PTCfg<64>::SMEM)
                     : go3(prefill_ptmem_kernel<__nv_bfloat16, 128>,
                           PTCfg<128>::SMEM);
    return D == 64 ? go3(prefill_ptmem_kernel<__half, 64>, PTCfg<64>::SMEM)
                   : go3(prefill_ptmem_kernel<__half, 128>, PTCfg<128>::SMEM);
  }
  if (bf16) {
    switch (D) {
      case 64:
        return go(prefill_pp_kernel<__nv_bfloat16, 64>, PPCfg<64>::SMEM,
                  PP_THREADS);
      case 128:
        return go(prefill_pp_kernel<__nv_bfloat16, 128>, PPCfg<128>::SMEM,
                  PP_THREADS);
      case 256:
        return go(prefill_tc_kernel<__nv_bfloat16, 256>, Cfg<256>::SMEM,
                  NUM_THREADS);
    }
  } else {
    switch (D) {
      case 64:
        return go(prefill_pp_kernel<__half, 64>, PPCfg<64>::SMEM, PP_THREADS);
      case 128:
        return go(prefill_pp_kernel<__half, 128>, PPCfg<128>::SMEM,
                  PP_THREADS);
      case 256:
        return go(prefill_tc_kernel<__half, 256>, Cfg<256>::SMEM, NUM_THREADS);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace pkv
