// Block-table attention on warp-level tensor-core MMA (mma.sync m16n8k16).
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (flash_attn_varlen_func with block_table, seqused_k, window_size,
// softcap, alibi_slopes, num_splits) and FlashAttentionMetadataBuilder (the
// packed-GQA handling for max_query_len = 1, and [num_splits, ...]
// intermediates for split-KV).
//
// One CTA owns (request b, KV head g, row tile, key split).  Query rows are
// packed (token, head-in-group): packed row R of request b is token R / G,
// query head g * G + R % G, so the G query heads that share a KV head share
// every K/V byte the CTA reads.  K/V pages are gathered through the block
// table with 16-byte cp.async copies into a STAGES-deep ring of shared-memory
// tiles (XOR-swizzled by 16-byte chunk so ldmatrix reads are conflict-free);
// keys at or beyond seqused_k are zero-filled, so uninitialised cache rows
// (even NaN) never reach the output.  Scores and P*V run on mma.sync with fp32
// accumulators, online softmax runs in base 2 in registers with quad shuffles.
//
// Two geometries are instantiated:
//   decode  (ROW_WARPS = 1, KEY_WARPS = 2..4): 16 packed rows, warps split the
//           keys of each tile, combined through shared memory at the end; with
//           a split plan each CTA covers one chunk of keys and writes fp32
//           partials (out, lse) that split_combine_kernel folds.
//   prefill (ROW_WARPS = 4, KEY_WARPS = 1): 64 packed rows, one warp per 16
//           rows over all keys (the first, non-tcgen05 prefill path).
#include <math.h>

#include "pkv_common.cuh"

// Decode geometry per head size.  D = 128: 2 stages of 64 keys, so three
// 100-KB-free CTAs (12 warps) share an SM; measured faster than 3 stages
// with two CTAs on the batched and long decode workloads.
#ifndef PKV_DECODE_STAGES_D128
#define PKV_DECODE_STAGES_D128 2
#endif
#ifndef PKV_DECODE_D256_KWARPS
#define PKV_DECODE_D256_KWARPS 2
#endif
#ifndef PKV_DECODE_D256_KT
#define PKV_DECODE_D256_KT 32
#endif
#ifndef PKV_DECODE_D256_STAGES
#define PKV_DECODE_D256_STAGES 2
#endif

namespace pkv {

template <int D, int ROW_WARPS, int KEY_WARPS, int KT, int STAGES,
          bool KV8 = false>
struct MmaCfg {
  static constexpr int NW = ROW_WARPS * KEY_WARPS;
  static constexpr int NT = NW * 32;
  static constexpr int ROWS = 16 * ROW_WARPS;
  static constexpr int KW = KT / KEY_WARPS;   // keys per warp per tile
  static constexpr int NKT = KW / 8;          // n8 tiles of S per warp
  static constexpr int CPR = D / 8;           // 16-byte chunks per row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int Q_BYTES = ROWS * ROW_BYTES;
  static constexpr int TILE_BYTES = KT * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int COMBINE_BYTES =
      KEY_WARPS > 1 ? KEY_WARPS * 16 * (D + 2) * 4 : 0;
  // fp8 cache: stages hold E4M3 tiles (1 byte per element); each tile is
  // converted into one 16-bit K/V work tile before the MMAs read it
  static constexpr int CPR8 = D / 16;         // 16-byte fp8 chunks per row
  static constexpr int STAGE8_BYTES = 2 * KT * D;
  static constexpr int RING_BYTES = KV8 ? STAGES * STAGE8_BYTES + STAGE_BYTES
                                        : STAGES * STAGE_BYTES;
  static constexpr int SMEM = Q_BYTES + RING_BYTES;
  static_assert(KW % 16 == 0, "each warp needs whole k16 steps of keys");
  static_assert(D % 64 == 0 || D == 64, "swizzle needs >= 8 chunks per row");
  static_assert(KEY_WARPS == 1 || ROW_WARPS == 1, "one split axis per CTA");
  static_assert(COMBINE_BYTES <= RING_BYTES, "combine buffer");
};

// Two E4M3 codes (low byte first) -> two 16-bit values of type T (exact).
template <typename T>
__device__ __forceinline__ uint32_t e4m3x2_to(uint16_t v);
template <>
__device__ __forceinline__ uint32_t e4m3x2_to<__half>(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}
template <>
__device__ __forceinline__ uint32_t e4m3x2_to<__nv_bfloat16>(uint16_t v) {
  const uint32_t h = e4m3x2_to<__half>(v);
  const __half2 hh = *reinterpret_cast<const __half2*>(&h);
  return pack2<__nv_bfloat16>(__low2float(hh), __high2float(hh));
}

template <typename T, int D, int ROW_WARPS, int KEY_WARPS, int KT, int STAGES,
          bool KV8 = false>
__global__ void __launch_bounds__(32 * ROW_WARPS * KEY_WARPS)
attn_mma_kernel(const AttnParams p) {
  // a prefill launch queued after this one in the same call may start
  // before this grid ends (it writes other requests' rows)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = MmaCfg<D, ROW_WARPS, KEY_WARPS, KT, STAGES, KV8>;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = (request, KV head) unit, y = row tile, z = split
  const int b = blockIdx.x / p.Hkv, g = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  const int G = p.G;
  const int q0 = p.cu_q[b];
  // rows past total_q (a cu_seqlens_q beyond the caller's buffers) are
  // never read or written
  const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
  const int koff = p.cu_k ? p.cu_k[b] : 0;      // non-paged: first key row
  const int L = p.cu_k ? p.cu_k[b + 1] - koff : p.seqused_k[b];
  if (q0 < 0 || q_len <= 0) return;
  const int rows = q_len * G;
  if (rows < p.min_rows || rows > p.max_rows) return;
  const int row0 = blockIdx.y * C::ROWS;
  if (row0 >= rows) return;
  const int row_end = min(rows, row0 + C::ROWS);

  int kmin, kmax;
  key_range(L, q_len, row0 / G, (row_end - 1) / G, p.causal, p.wl, p.wr, kmin,
            kmax);
  int lo = kmin, hi = kmax;
  if (p.chunk > 0) {
    // The grid has gridDim.z splits; if the caller's max_seqlen_k was too
    // small for this request, the last split takes the rest of the range.
    const int nsplit = split_count(kmin, kmax, p.chunk, gridDim.z);
    if (static_cast<int>(blockIdx.z) >= nsplit) return;
    split_bounds(kmin, kmax, p.chunk, nsplit, blockIdx.z, lo, hi);
  }
  // Keys are only followed through the table while it has entries.
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  const int L_tab = p.cu_k ? (koff < 0 ? 0 : max(0, min(L, p.total_k - koff)))
                           : min(L, p.max_blocks * p.BS);
  if (L_tab < L && tid == 0 && blockIdx.z == 0 && blockIdx.y == 0)
    atomicOr(p.err, kErrBadTable);

  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ KC = static_cast<const T*>(p.kc);
  const T* __restrict__ VC = static_cast<const T*>(p.vc);
  const int32_t* __restrict__ bt = p.block_table + b * p.bt_stride;

  unsigned char* sQ = smem;
  unsigned char* sKV = smem + C::Q_BYTES;
  const uint32_t sQ_u = smem_u32(sQ);
  const uint32_t sKV_u = smem_u32(sKV);

  // ---- Q tile: packed rows row0 .. row0 + ROWS (zero past row_end)
  for (int i = tid; i < C::ROWS * C::CPR; i += C::NT) {
    const int r = i / C::CPR, ch = i - (i / C::CPR) * C::CPR;
    const int R = row0 + r;
    const bool ok = R < row_end;
    const T* src = Q;
    if (ok) {
      const int tok = q0 + R / G, h = g * G + R % G;
      src = Q + static_cast<int64_t>(tok) * p.q_st +
            static_cast<int64_t>(h) * p.q_sh + ch * 8;
    }
    cp_async_16(sQ_u + swz<C::ROW_BYTES>(r, ch), src, ok ? 16 : 0);
  }

  const int n_tiles = (hi - lo + KT - 1) / KT;
  // Page ids travel through a small shared ring: the ids of tile t are
  // fetched from the block table (global) one iteration before the tile's
  // copies are issued, so table latency never sits in front of a copy.
  constexpr int PPT = KT / 16 + 1;              // pages a tile can touch
  constexpr int RING = STAGES + 1;
  __shared__ int s_pg[RING][PPT];
  const int bs_shift = p.bs_shift;
  auto page_index = [&](int j) { return bs_shift >= 0 ? (j >> bs_shift)
                                                       : j / p.BS; };
  auto fetch_id = [&](int t) -> int {           // id of page `tid` of tile t
    if (t >= n_tiles || tid >= PPT || p.cu_k) return -1;
    const int kt = lo + t * KT;
    const int jb = page_index(kt) + tid;
    if (jb * p.BS >= min(L_tab, kt + KT)) return -1;
    const int blk = __ldg(bt + jb);
    if (blk < 0 || blk >= p.num_blocks) {
      atomicOr(p.err, kErrBadBlock);
      return -1;
    }
    return blk;
  };
  auto load_tile = [&](int it, int stage) {
    const int kt = lo + it * KT;
    const int jb0 = page_index(kt);
    const int* pg = s_pg[it % RING];
    if constexpr (KV8) {
      // E4M3 rows, D bytes each, unswizzled (read once by the converter)
      const uint32_t sK8 = sKV_u + stage * C::STAGE8_BYTES;
      const uint32_t sV8 = sK8 + KT * D;
      const unsigned char* K8 = static_cast<const unsigned char*>(p.kc);
      const unsigned char* V8 = static_cast<const unsigned char*>(p.vc);
#pragma unroll 4
      for (int i = tid; i < KT * C::CPR8; i += C::NT) {
        const int r = i / C::CPR8, ch = i - (i / C::CPR8) * C::CPR8;
        const int j = kt + r;
        const int jb = p.cu_k ? 0 : page_index(j);
        const int blk = j < L_tab ? (p.cu_k ? 0 : pg[jb - jb0]) : -1;
        const bool ok = blk >= 0;
        int64_t off = 0;
        if (ok)
          off = static_cast<int64_t>(blk) * p.c_sb +
                static_cast<int64_t>(p.cu_k ? koff + j : j - jb * p.BS) * p.c_sr +
                static_cast<int64_t>(g) * p.c_sh + ch * 16;
        cp_async_16(sK8 + r * D + ch * 16, K8 + off, ok ? 16 : 0);
        cp_async_16(sV8 + r * D + ch * 16, V8 + off, ok ? 16 : 0);
      }
      return;
    }
    const uint32_t sK = sKV_u + stage * C::STAGE_BYTES;
    const uint32_t sV = sK + C::TILE_BYTES;
#pragma unroll 4
    for (int i = tid; i < KT * C::CPR; i += C::NT) {
      const int r = i / C::CPR, ch = i - (i / C::CPR) * C::CPR;
      const int j = kt + r;
      const int jb = p.cu_k ? 0 : page_index(j);
      const int blk = j < L_tab ? (p.cu_k ? 0 : pg[jb - jb0]) : -1;
      const bool ok = blk >= 0;
      int64_t off = 0;
      if (ok)
        off = static_cast<int64_t>(blk) * p.c_sb +
              static_cast<int64_t>(p.cu_k ? koff + j : j - jb * p.BS) * p.c_sr +
              static_cast<int64_t>(g) * p.c_sh + ch * 8;
      const uint32_t d = swz<C::ROW_BYTES>(r, ch);
      cp_async_16(sK + d, KC + off, ok ? 16 : 0);
      cp_async_16(sV + d, VC + off, ok ? 16 : 0);
    }
  };

  for (int t = 0; t < STAGES; ++t) {
    const int id = fetch_id(t);
    if (tid < PPT) s_pg[t % RING][tid] = id;
  }
  __syncthreads();
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  // ---- per-thread row bookkeeping
  const int wrow = (KEY_WARPS == 1) ? warp : 0;   // row-warp index
  const int wkey = (KEY_WARPS == 1) ? 0 : warp;   // key-warp index
  const int g8 = lane >> 2, c4 = lane & 3;
  const int rA = row0 + wrow * 16 + g8, rB = rA + 8;
  const int ctx = L - q_len;
  const int pA = ctx + rA / G, pB = ctx + rB / G;
  const bool okA = rA < row_end, okB = rB < row_end;
  float slopeA = 0.f, slopeB = 0.f;
  if (p.alibi) {
    if (okA) slopeA = p.alibi[g * G + rA % G];
    if (okB) slopeB = p.alibi[g * G + rB % G];
  }
  const bool plain = (p.softcap <= 0.f) && (p.alibi == nullptr);
  // soft-cap without ALiBi: interior tiles need only the capped logit
  const bool capped = (p.softcap > 0.f) && (p.alibi == nullptr);
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
  // fp8 cache: value = code * scale, so k_scale joins the logit scale and
  // v_scale multiplies the output
  const float kscale = p.k_scale ? *p.k_scale : 1.f;
  const float vscale = p.v_scale ? *p.v_scale : 1.f;
  const float qk_scale = p.scale * kscale;
  const float scale_log2 = qk_scale * kLog2e;
  // keys every valid row of this CTA admits: tiles inside [full_lo,
  // full_hi) skip the per-key mask (rows past row_end are never stored)
  int full_lo = lo, full_hi = hi;
  {
    const int p_lo = ctx + row0 / G, p_hi = ctx + (row_end - 1) / G;
    if (p.wl >= 0) full_lo = max(full_lo, p_hi - p.wl);
    if (p.causal) full_hi = min(full_hi, p_lo + 1);
    if (p.wr >= 0) full_hi = min(full_hi, p_lo + p.wr + 1);
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  // ldmatrix lane geometry
  const int lm_mi = lane >> 3, lm_r = lane & 7;

  for (int it = 0; it < n_tiles; ++it) {
    const int next_id = fetch_id(it + STAGES);    // lands in the ring below
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nxt = it + STAGES - 1;
      if (nxt < n_tiles) load_tile(nxt, nxt % STAGES);
      cp_async_commit();
    }
    const int stage = it % STAGES;
    uint32_t sK = sKV_u + stage * C::STAGE_BYTES;
    uint32_t sV = sK + C::TILE_BYTES;
    if constexpr (KV8) {
      // E4M3 stage -> 16-bit work tile (exact; the scales are applied to
      // the logits and to the output instead)
      const uint32_t sK8 = sKV_u + stage * C::STAGE8_BYTES;
      const uint32_t sW = sKV_u + STAGES * C::STAGE8_BYTES;
      for (int i = tid; i < 2 * KT * C::CPR8; i += C::NT) {
        const int mat = i / (KT * C::CPR8);
        const int rem = i - mat * (KT * C::CPR8);
        const int r = rem / C::CPR8, ch = rem - (rem / C::CPR8) * C::CPR8;
        uint4 raw;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                     : "r"(sK8 + mat * KT * D + r * D + ch * 16));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          o[2 * q] = e4m3x2_to<T>(static_cast<uint16_t>(w[q] & 0xFFFF));
          o[2 * q + 1] = e4m3x2_to<T>(static_cast<uint16_t>(w[q] >> 16));
        }
        const uint32_t dst = sW + mat * C::TILE_BYTES;
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         dst + swz<C::ROW_BYTES>(r, 2 * ch)),
                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]));
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         dst + swz<C::ROW_BYTES>(r, 2 * ch + 1)),
                     "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]));
      }
      __syncthreads();
      sK = sW;
      sV = sW + C::TILE_BYTES;
    }
    const int kw0 = wkey * C::KW;          // first key of this warp in tile
    const int kt = lo + it * KT;

    // S = Q K^T for this warp's 16 rows x KW keys
    float s[C::NKT][4];
#pragma unroll
    for (int i = 0; i < C::NKT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      {
        const int r = wrow * 16 + lm_r + (lm_mi & 1) * 8;
        const int ch = kk * 2 + (lm_mi >> 1);
        ldmatrix_x4(sQ_u + swz<C::ROW_BYTES>(r, ch), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int np = 0; np < C::NKT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        const int r = kw0 + np * 16 + lm_r + (lm_mi >> 1) * 8;
        const int ch = kk * 2 + (lm_mi & 1);
        ldmatrix_x4(sK + swz<C::ROW_BYTES>(r, ch), b0, b1, b2, b3);
        mma_16816<T>(s[2 * np], a, b0, b1);
        mma_16816<T>(s[2 * np + 1], a, b2, b3);
      }
    }

    // logits (base 2) with masks
    float mxA = -INFINITY, mxB = -INFINITY;
    const bool interior = kt >= full_lo && kt + KT <= full_hi;
    if (plain && interior) {
#pragma unroll
      for (int nt = 0; nt < C::NKT; ++nt) {
        s[nt][0] *= scale_log2;
        s[nt][1] *= scale_log2;
        s[nt][2] *= scale_log2;
        s[nt][3] *= scale_log2;
        mxA = fmaxf(mxA, fmaxf(s[nt][0], s[nt][1]));
        mxB = fmaxf(mxB, fmaxf(s[nt][2], s[nt][3]));
      }
    } else if (capped && interior) {
      const float pre = qk_scale * inv_cap, post = p.softcap * kLog2e;
#pragma unroll
      for (int nt = 0; nt < C::NKT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = post * tanh_fast(s[nt][e] * pre);
        mxA = fmaxf(mxA, fmaxf(s[nt][0], s[nt][1]));
        mxB = fmaxf(mxB, fmaxf(s[nt][2], s[nt][3]));
      }
    } else {
#pragma unroll
    for (int nt = 0; nt < C::NKT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kt + kw0 + nt * 8 + 2 * c4 + (e & 1);
        const bool rowB = e >= 2;
        const int pos = rowB ? pB : pA;
        float x = s[nt][e];
        if (plain) {
          x *= scale_log2;
        } else {
          x *= qk_scale;
          if (p.softcap > 0.f) x = p.softcap * tanh_fast(x * inv_cap);
          if (p.alibi) x -= (rowB ? slopeB : slopeA) * fabsf(float(pos - key));
          x *= kLog2e;
        }
        bool ok = (rowB ? okB : okA) && key >= lo && key < hi;
        if (p.causal) ok = ok && key <= pos;
        if (p.wl >= 0) ok = ok && key >= pos - p.wl;
        if (p.wr >= 0) ok = ok && key <= pos + p.wr;
        x = ok ? x : -INFINITY;
        s[nt][e] = x;
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
      s[nt][0] = ex2(s[nt][0] - baseA);
      s[nt][1] = ex2(s[nt][1] - baseA);
      s[nt][2] = ex2(s[nt][2] - baseB);
      s[nt][3] = ex2(s[nt][3] - baseB);
      sumA += s[nt][0] + s[nt][1];
      sumB += s[nt][2] + s[nt][3];
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
    // O += P V
#pragma unroll
    for (int ks = 0; ks < C::KW / 16; ++ks) {
      uint32_t a[4];
      a[0] = pack2<T>(s[2 * ks][0], s[2 * ks][1]);
      a[1] = pack2<T>(s[2 * ks][2], s[2 * ks][3]);
      a[2] = pack2<T>(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      a[3] = pack2<T>(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        const int r = kw0 + ks * 16 + lm_r + (lm_mi & 1) * 8;
        const int ch = dp * 2 + (lm_mi >> 1);
        ldmatrix_x4_trans(sV + swz<C::ROW_BYTES>(r, ch), b0, b1, b2, b3);
        mma_16816<T>(o[2 * dp], a, b0, b1);
        mma_16816<T>(o[2 * dp + 1], a, b2, b3);
      }
    }
    if (tid < PPT) s_pg[(it + STAGES) % RING][tid] = next_id;
  }
  cp_async_wait<0>();

  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);

  const bool split = p.chunk > 0;
  T* __restrict__ OUT = static_cast<T*>(p.out);

  if constexpr (KEY_WARPS == 1) {
    // each warp owns its 16 rows: write straight from the fragments
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? rB : rA;
      if (r >= row_end) continue;
      const float l = half ? lB : lA, m = half ? mB : mA;
      const int tok = q0 + r / G, h = g * G + r % G;
      float inv, lse;   // a sink enters once: here, or in the split combine
      finish_row(m, l, split ? nullptr : p.sinks, h, &inv, &lse);
      inv *= vscale;
      if (!split) {
        T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
                 static_cast<int64_t>(h) * p.o_sh;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<uint32_t*>(dst + dn * 8 + 2 * c4) =
              pack2<T>(o[dn][2 * half] * inv, o[dn][2 * half + 1] * inv);
        if (p.lse && c4 == 0) p.lse[static_cast<int64_t>(h) * p.total_q + tok] = lse;
      } else {
        float* dst = p.part_o +
                     ((static_cast<int64_t>(blockIdx.z) * p.part_rows +
                       part_row(p.part_tpr, b, q0, tok)) *
                          p.Hq + h) * D;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<float2*>(dst + dn * 8 + 2 * c4) =
              make_float2(o[dn][2 * half] * inv, o[dn][2 * half + 1] * inv);
        if (c4 == 0)
          p.part_lse[(static_cast<int64_t>(blockIdx.z) * p.Hq + h) *
                         p.part_rows +
                     part_row(p.part_tpr, b, q0, tok)] = lse;
      }
    }
  } else {
    // combine the key-warps' partial states through shared memory
    __syncthreads();
    float* sm_ml = reinterpret_cast<float*>(sKV);           // [KW][16][2]
    float* sm_o = sm_ml + KEY_WARPS * 16 * 2;               // [KW][16][D]
    if (c4 == 0) {
      sm_ml[(wkey * 16 + g8) * 2 + 0] = mA;
      sm_ml[(wkey * 16 + g8) * 2 + 1] = lA;
      sm_ml[(wkey * 16 + g8 + 8) * 2 + 0] = mB;
      sm_ml[(wkey * 16 + g8 + 8) * 2 + 1] = lB;
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      *reinterpret_cast<float2*>(sm_o + (wkey * 16 + g8) * D + dn * 8 +
                                 2 * c4) = make_float2(o[dn][0], o[dn][1]);
      *reinterpret_cast<float2*>(sm_o + (wkey * 16 + g8 + 8) * D + dn * 8 +
                                 2 * c4) = make_float2(o[dn][2], o[dn][3]);
    }
    __syncthreads();
    for (int i = tid; i < 16 * (D / 4); i += C::NT) {
      const int rr = i / (D / 4), c = (i - rr * (D / 4)) * 4;
      const int R = row0 + rr;
      if (R >= row_end) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < KEY_WARPS; ++w)
        M = fmaxf(M, sm_ml[(w * 16 + rr) * 2]);
      const float base = (M == -INFINITY) ? 0.f : M;
      float lsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < KEY_WARPS; ++w) {
        const float f = ex2(sm_ml[(w * 16 + rr) * 2] - base);
        lsum += f * sm_ml[(w * 16 + rr) * 2 + 1];
        const float4 v = *reinterpret_cast<const float4*>(
            sm_o + (w * 16 + rr) * D + c);
        acc.x += f * v.x;
        acc.y += f * v.y;
        acc.z += f * v.z;
        acc.w += f * v.w;
      }
      const int tok = q0 + R / G, h = g * G + R % G;
      float inv, lse;   // a sink enters once: here, or in the split combine
      finish_row(M, lsum, split ? nullptr : p.sinks, h, &inv, &lse);
      inv *= vscale;
      if (!split) {
        T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
                 static_cast<int64_t>(h) * p.o_sh + c;
        uint2 pk;
        pk.x = pack2<T>(acc.x * inv, acc.y * inv);
        pk.y = pack2<T>(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(dst) = pk;
        if (p.lse && c == 0) p.lse[static_cast<int64_t>(h) * p.total_q + tok] = lse;
      } else {
        float* dst = p.part_o +
                     ((static_cast<int64_t>(blockIdx.z) * p.part_rows +
                       part_row(p.part_tpr, b, q0, tok)) *
                          p.Hq + h) * D + c;
        *reinterpret_cast<float4*>(dst) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (c == 0)
          p.part_lse[(static_cast<int64_t>(blockIdx.z) * p.Hq + h) *
                         p.part_rows +
                     part_row(p.part_tpr, b, q0, tok)] = lse;
      }
    }
  }
}

// Fold the split-KV partials of decode-class requests: one warp per
// (request, query head), looping over the request's tokens.
template <typename T>
__global__ void __launch_bounds__(128)
split_combine_kernel(const CombineParams p) {
  // a prefill launch queued after this one in the same call may start
  // before this grid ends (it writes other requests' rows)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // launched as a programmatic dependent of the decode grid: its partials
  // are complete and visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + warp;
  const int b = blockIdx.x;
  if (h >= p.Hq) return;
  const int q0 = p.cu_q[b];
  const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
  if (q0 < 0 || q_len <= 0) return;
  const int rows = q_len * p.G;
  if (rows < p.min_rows || rows > p.max_rows) return;
  const int L = p.cu_k ? p.cu_k[b + 1] - p.cu_k[b] : p.seqused_k[b];
  int kmin, kmax;
  key_range(L, q_len, 0, q_len - 1, p.causal, p.wl, p.wr, kmin, kmax);
  const int nsplit = split_count(kmin, kmax, p.chunk, p.splits);
  const int D = p.D;
  T* __restrict__ OUT = static_cast<T*>(p.out);
  for (int i = 0; i < q_len; ++i) {
    const int tok = q0 + i;
    const int64_t prow = part_row(p.part_tpr, b, q0, tok);
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32)
      M = fmaxf(M, p.part_lse[(static_cast<int64_t>(s) * p.Hq + h) *
                                  p.part_rows + prow]);
#pragma unroll
    for (int o = 16; o; o >>= 1)
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // a sink logit is one more softmax term without a value
    const float sink = p.sinks ? p.sinks[h] : -INFINITY;
    M = fmaxf(M, sink);
    const float base = (M == -INFINITY) ? 0.f : M;
    const float w_sink = p.sinks ? __expf(sink - base) : 0.f;
    float lsum = w_sink;
    for (int c = lane * 4; c < D; c += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float ls = w_sink;
      for (int s = 0; s < nsplit; ++s) {
        const float l = p.part_lse[(static_cast<int64_t>(s) * p.Hq + h) *
                                       p.part_rows + prow];
        const float w = (l == -INFINITY) ? 0.f : __expf(l - base);
        ls += w;
        if (w != 0.f) {
          const float4 v = *reinterpret_cast<const float4*>(
              p.part_o +
              ((static_cast<int64_t>(s) * p.part_rows + prow) * p.Hq + h) * D +
              c);
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
      }
      lsum = ls;
      const float inv = ls > 0.f ? 1.f / ls : 0.f;
      T* dst = OUT + static_cast<int64_t>(tok) * p.o_st +
               static_cast<int64_t>(h) * p.o_sh + c;
      uint2 pk;
      pk.x = pack2<T>(acc.x * inv, acc.y * inv);
      pk.y = pack2<T>(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    }
    if (p.lse && lane == 0) {
      // every lane of the warp saw the same weights; lane 0 has c = 0
      p.lse[static_cast<int64_t>(h) * p.total_q + tok] =
          lsum > 0.f ? base + __logf(lsum) : -INFINITY;
    }
  }
}

// ------------------------------------------------------------------ launch

template <typename T, int D, int RW, int KWp, int KT, int ST,
          bool KV8 = false>
static cudaError_t launch_cfg(const AttnParams& p, dim3 grid,
                              cudaStream_t stream) {
  using C = MmaCfg<D, RW, KWp, KT, ST, KV8>;
  auto kern = attn_mma_kernel<T, D, RW, KWp, KT, ST, KV8>;
  cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  note_launch();
  kern<<<grid, C::NT, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t decode_dispatch(const AttnParams& p, int D, dim3 grid,
                                   cudaStream_t s) {
  if (p.kv_fp8) {
    switch (D) {
      case 64:  return launch_cfg<T, 64, 1, 4, kDecodeKT, 4, true>(p, grid, s);
      case 128: return launch_cfg<T, 128, 1, 4, kDecodeKT, 2, true>(p, grid, s);
      case 256: return launch_cfg<T, 256, 1, 2, 32, 2, true>(p, grid, s);
      default:  return cudaErrorInvalidValue;
    }
  }
  switch (D) {
    case 64:  return launch_cfg<T, 64, 1, 4, kDecodeKT, 4>(p, grid, s);
    case 128: return launch_cfg<T, 128, 1, 4, kDecodeKT, PKV_DECODE_STAGES_D128>(p, grid, s);
    case 256: return launch_cfg<T, 256, 1, PKV_DECODE_D256_KWARPS,
                                PKV_DECODE_D256_KT, PKV_DECODE_D256_STAGES>(
        p, grid, s);
    default:  return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t prefill_dispatch(const AttnParams& p, int D, dim3 grid,
                                    cudaStream_t s) {
  switch (D) {
    case 64:  return launch_cfg<T, 64, 4, 1, 64, 3>(p, grid, s);
    case 128: return launch_cfg<T, 128, 4, 1, 64, 2>(p, grid, s);
    case 256: return launch_cfg<T, 256, 4, 1, 32, 2>(p, grid, s);
    default:  return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_attn(const AttnParams& p, int D, bool bf16,
                               int grid_x, int grid_y, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(p.batch) * p.Hkv, grid_y, grid_x);
  return bf16 ? decode_dispatch<__nv_bfloat16>(p, D, grid, stream)
              : decode_dispatch<__half>(p, D, grid, stream);
}

cudaError_t launch_prefill_attn_mma(const AttnParams& p, int D, bool bf16,
                                    int grid_y, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(p.batch) * p.Hkv, grid_y, 1);
  return bf16 ? prefill_dispatch<__nv_bfloat16>(p, D, grid, stream)
              : prefill_dispatch<__half>(p, D, grid, stream);
}

cudaError_t launch_split_combine(const CombineParams& p, bool bf16,
                                 cudaStream_t stream, bool pdl) {
  dim3 grid(static_cast<unsigned>(p.batch), (p.Hq + 3) / 4);
  note_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e =
      bf16 ? cudaLaunchKernelEx(&cfg, split_combine_kernel<__nv_bfloat16>, p)
           : cudaLaunchKernelEx(&cfg, split_combine_kernel<__half>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
