// Decode attention with TMA page loads and a producer warp.
//
// Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
// forward (flash_attn_varlen_func over the paged cache: cu_seqlens_q,
// seqused_k, block_table, causal, window_size, softcap, alibi_slopes, LSE)
// and FlashAttentionMetadataBuilder (split-KV decoding of requests with one
// query per KV-head group, intermediates of [num_splits, ...] combined by
// LSE).  Same math as the cp.async decode kernel in attn_mma.cu; this one
// moves K/V with the tensor-memory accelerator.
//
// One CTA owns (request b, KV head g, split s).  Its rows are the request's
// q_len * G <= 16 packed (token, head-in-group) query rows, the M dimension
// of mma.sync m16n8k16 (a 16 x KT x D contraction is far too small for a
// 128-row tcgen05 tile; the kernel is bound by HBM, not by the MMAs).
//
//   warp NCW (producer)  lane i fetches the page id of box i of the next
//                        tile from the block table, then issues the tile's
//                        K and V boxes (128-byte swizzle) into a
//                        STAGES-deep ring; K and V complete on separate
//                        mbarriers.  A box is RB rows x 64 columns
//                        (cp.async.bulk.tensor.4d), or at D = 128 over
//                        views that allow it one row-group box holding
//                        both column blocks of the page's RB rows (5-D),
//                        or for an E4M3 cache RB rows x 128 one-byte codes
//   warps 0..NCW-1       each owns KW = KT / NCW keys of every tile:
//                        S = Q K^T, online softmax (base 2), O += P V, then
//                        releases the stage; at the end the warps' partial
//                        states are merged through shared memory
//
// E4M3 caches (D = 128): the MMAs run on f16; Q becomes f16 A fragments
// once per CTA (a bf16 query scaled by a power of two, exact in f16), and
// the K and V code fragments convert in registers after their ldmatrix
// (k_scale joins the logit scale, v_scale the output).
//
// Tiles start on KT-key boundaries, so every box starts on a page boundary
// multiple of RB (RB divides both block_size and KT).  Keys outside the
// split's [lo, hi) are masked; V rows at or past the end of the loaded range
// are zeroed before P V (they may hold another request's NaN padding).
// Every mbarrier wait is bounded (kWaitLimitNs); a CTA whose wait runs out
// records kErrTimeout, drains the copies it issued and exits without
// writing.
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "pkv_common.cuh"
#include "tma_util.cuh"

namespace pkv {
namespace dtma {

template <int D, int NCW, int KT, int STAGES, bool KV8 = false>
struct Cfg {
  static constexpr int NT = (NCW + 1) * 32;     // consumers + producer warp
  static constexpr int CT = NCW * 32;           // consumer threads
  static constexpr int KW = KT / NCW;           // keys per warp per tile
  static constexpr int NKT = KW / 8;            // n8 tiles of S per warp
  static constexpr int BOXC = KV8 ? 128 : 64;   // columns per TMA box
  static constexpr int NCB = D / BOXC;          // 128-byte column blocks
  static constexpr int CPR = D / 8;             // 16-byte chunks per Q row
  static constexpr int RCH = KV8 ? D / 16 : D / 8;   // ... per K/V row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int CB_BYTES = KT * 128;     // one column block of a tile
  static constexpr int TILE_BYTES = NCB * CB_BYTES;
  static constexpr int RING_BYTES = STAGES * 2 * TILE_BYTES;
  static constexpr int Q_BYTES = 16 * ROW_BYTES;
  // E4M3 caches: f16 A fragments of Q per k16 step (32 lanes x 16 bytes),
  // and the consumer warps' largest |q|
  static constexpr int QFRAG_BYTES = KV8 ? (D / 16) * 32 * 16 : 0;
  static constexpr int QMAX_BYTES = KV8 ? 16 * ((NCW * 4 + 15) / 16) : 0;
  static constexpr int OFF_Q = RING_BYTES;
  static constexpr int OFF_QFRAG = OFF_Q + Q_BYTES;
  static constexpr int OFF_QMAX = OFF_QFRAG + QFRAG_BYTES;
  static constexpr int OFF_BAR = OFF_QMAX + QMAX_BYTES;
  static constexpr int BAR_BYTES = 3 * STAGES * 8 + 8 + 4 * STAGES;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;   // + alignment
  static constexpr int COMBINE_BYTES = NCW * 16 * (D + 2) * 4;
  static_assert(KW % 16 == 0, "each warp needs whole k16 steps of keys");
  static_assert(D % BOXC == 0, "whole TMA boxes per row");
  static_assert(!KV8 || NKT == 2 || NKT == 4, "ldmatrix grouping of codes");
  static_assert(CB_BYTES % 1024 == 0, "128-byte swizzle atoms");
  static_assert(COMBINE_BYTES <= RING_BYTES, "combine buffer");
};

// Byte offset of 16-byte chunk `ch` (0 .. D/8-1) of row r in a K/V tile
// with the 128-byte swizzle: [column block][key][64] from 4-D boxes (RG
// false), [8-key group][column block][8 keys][64] from row-group boxes.
template <int KT, int D, bool RG>
__device__ __forceinline__ uint32_t kv_off(int r, int ch) {
  if constexpr (RG)
    return static_cast<uint32_t>((r >> 3) * (D / 64 * 1024) +
                                 (ch >> 3) * 1024) +
           sw128(r & 7, ch & 7);
  else
    return static_cast<uint32_t>((ch >> 3) * (KT * 128)) + sw128(r, ch & 7);
}

template <typename T, int D, int NCW, int KT, int STAGES, bool RG, bool KV8>
__device__ __forceinline__ void decode_tma_body(const AttnParams& p,
                                                const CUtensorMap& tm_k,
                                                const CUtensorMap& tm_v) {
  using C = Cfg<D, NCW, KT, STAGES, KV8>;
  // E4M3 caches: the MMAs run on f16 (codes convert to f16 exactly)
  using MT = typename std::conditional<KV8, __half, T>::type;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_u - raw_u);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = (request, KV head) unit, y = split
  const int b = blockIdx.x / p.Hkv, g = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  const int G = p.G;
  const int q0 = p.cu_q[b];
  const int q_len = min(p.cu_q[b + 1] - q0, p.total_q - q0);
  if (q0 < 0 || q_len <= 0) return;
  const int rows = q_len * G;
  if (rows < p.min_rows || rows > p.max_rows || rows > 16) return;
  const int koff = p.cu_k ? p.cu_k[b] : 0;      // non-paged: first key row
  const int L = p.cu_k ? p.cu_k[b + 1] - koff : p.seqused_k[b];
  // rows past the table (or, non-paged, past the K/V tensor) are not read
  const int L_tab = p.cu_k ? (koff < 0 ? 0 : max(0, min(L, p.total_k - koff)))
                           : min(L, p.max_blocks * p.BS);
  if (L_tab < L && tid == 0 && blockIdx.y == 0)
    atomicOr(p.err, kErrBadTable);

  int kmin, kmax;
  key_range(L, q_len, 0, q_len - 1, p.causal, p.wl, p.wr, kmin, kmax);
  int lo = kmin, hi = kmax;
  if (p.chunk > 0) {
    const int nsplit = split_count(kmin, kmax, p.chunk, gridDim.y);
    if (static_cast<int>(blockIdx.y) >= nsplit) return;
    split_bounds(kmin, kmax, p.chunk, nsplit, blockIdx.y, lo, hi);
  }
  hi = min(hi, L_tab);
  const int kt0 = (lo / KT) * KT;
  const int n_tiles = hi > lo ? (hi - kt0 + KT - 1) / KT : 0;
  const int RB = p.rb;                          // rows per box

  const uint32_t ring = base_u;
  const uint32_t sQ = base_u + C::OFF_Q;
  const uint32_t bar0 = base_u + C::OFF_BAR;
  auto full_k = [&](int s) { return bar0 + 8 * s; };
  auto full_v = [&](int s) { return bar0 + 8 * (STAGES + s); };
  auto empty = [&](int s) { return bar0 + 8 * (2 * STAGES + s); };
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(base + C::OFF_BAR + 3 * STAGES * 8);
  // per stage: boxes of the tile whose page id was out of range (not
  // loaded; their K and V rows are zeroed by the consumers instead)
  volatile unsigned* bad_boxes = reinterpret_cast<volatile unsigned*>(
      base + C::OFF_BAR + 3 * STAGES * 8 + 8);
  auto tile_k = [&](int s) { return ring + s * 2 * C::TILE_BYTES; };
  auto tile_v = [&](int s) { return ring + s * 2 * C::TILE_BYTES + C::TILE_BYTES; };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_k(s), 1);
      mbar_init(full_v(s), 1);
      mbar_init(empty(s), NCW);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp < NCW) {
    // ---- Q tile: packed rows 0 .. 16 (zero past rows)
    const T* Q = static_cast<const T*>(p.q);
    for (int i = tid; i < 16 * C::CPR; i += C::CT) {
      const int r = i / C::CPR, ch = i - (i / C::CPR) * C::CPR;
      const bool ok = r < rows;
      const T* src = Q;
      if (ok)
        src = Q + static_cast<int64_t>(q0 + r / G) * p.q_st +
              static_cast<int64_t>(g * G + r % G) * p.q_sh + ch * 8;
      cp_async_16(sQ + swz<C::ROW_BYTES>(r, ch), src, ok ? 16 : 0);
    }
    cp_async_commit();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    if (n_tiles == 0) return;
    const int nb_max = KT / RB;
    // K/V pages are read once: their L2 lines go first (measured on GB300:
    // batched decode 0.1148 -> 0.1116 ms, long decode 0.654 -> 0.649 ms,
    // cascade 0.1357 -> 0.1342 ms against plain loads)
    const uint64_t pol = l2_evict_first_policy();
    auto kv_load = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1,
                       int c2, int c3, uint32_t bar) {
      tma_load_4d_hint(dst, m, c0, c1, c2, c3, bar, pol);
    };
    const int32_t* bt = p.cu_k ? nullptr
                               : p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    auto fetch = [&](int t) -> int {            // page id of box `lane`
      const int k0 = kt0 + t * KT + lane * RB;
      if (t >= n_tiles || lane >= nb_max || k0 >= hi || !bt) return 0;
      const int blk = __ldg(bt + k0 / p.BS);
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.err, kErrBadBlock);
        return -1;
      }
      return blk;
    };
    int issued = 0;
    int cur = fetch(0);
    for (int t = 0; t < n_tiles; ++t) {
      const int nxt = fetch(t + 1);
      const int s = t % STAGES;
      const int kt = kt0 + t * KT;
      int nbox = (hi - kt + RB - 1) / RB;
      if (nbox > nb_max) nbox = nb_max;
      const unsigned bad = __ballot_sync(0xffffffffu, lane < nbox && cur < 0);
      int stop = 0;
      if (lane == 0) {
        if (t >= STAGES &&
            !mbar_wait_lim(empty(s), ((t / STAGES) - 1) & 1, abort_flag,
                        p.err, p.wait_ns)) {
          stop = 1;
        } else {
          bad_boxes[s] = bad;
          const uint32_t bytes = (nbox - __popc(bad)) * C::NCB * RB * 128;
          mbar_expect_tx(full_k(s), bytes);
          mbar_expect_tx(full_v(s), bytes);
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (stop) break;
      if (RG && lane < nbox && cur >= 0) {
        // one row-group box per page and matrix
        const int row = (kt + lane * RB) % p.BS;
        const uint32_t off = lane * RB * (C::NCB * 128);
        if (p.kv_order_hnd) {
          tma_load_5d_hint(tile_k(s) + off, &tm_k, 0, 0, 0, row >> 3,
                           cur * p.Hkv + g, full_k(s), pol);
          tma_load_5d_hint(tile_v(s) + off, &tm_v, 0, 0, 0, row >> 3,
                           cur * p.Hkv + g, full_v(s), pol);
        } else {
          const int grp = cur * (p.BS >> 3) + (row >> 3);
          tma_load_5d_hint(tile_k(s) + off, &tm_k, 0, 0, 0, grp, g,
                           full_k(s), pol);
          tma_load_5d_hint(tile_v(s) + off, &tm_v, 0, 0, 0, grp, g,
                           full_v(s), pol);
        }
      } else if (lane < nbox && cur >= 0) {
        const int k0 = kt + lane * RB;
        const int row = p.cu_k ? koff + k0 : k0 % p.BS;
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb) {
          const uint32_t dst = tile_k(s) + cb * C::CB_BYTES + lane * RB * 128;
          if (p.kv_order_hnd)
            kv_load(dst, &tm_k, cb * C::BOXC, row, g, cur, full_k(s));
          else
            kv_load(dst, &tm_k, cb * C::BOXC, g, row, cur, full_k(s));
        }
#pragma unroll
        for (int cb = 0; cb < C::NCB; ++cb) {
          const uint32_t dst = tile_v(s) + cb * C::CB_BYTES + lane * RB * 128;
          if (p.kv_order_hnd)
            kv_load(dst, &tm_v, cb * C::BOXC, row, g, cur, full_v(s));
          else
            kv_load(dst, &tm_v, cb * C::BOXC, g, row, cur, full_v(s));
        }
      }
      issued = t + 1;
      cur = nxt;
    }
    if (lane == 0) {
      // no copy of this CTA may still be in flight when it exits (the
      // consumers wait for every tile, unless a wait ran out)
      for (int t = max(0, issued - STAGES); t < issued; ++t) {
        mbar_drain(full_k(t % STAGES), (t / STAGES) & 1);
        mbar_drain(full_v(t % STAGES), (t / STAGES) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  cp_async_wait<0>();
  asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");
  // E4M3 cache: Q as f16 A fragments in the head-dimension order the K
  // code fragments arrive in (d = 16 ks + 4 c4 + {0,1} in registers 0/1,
  // + {2,3} in registers 2/3).  A bf16 query is scaled by the power of two
  // that puts its largest magnitude in [2^14, 2^15), so every value is
  // exact in f16; the factor joins the logit scale.
  const uint32_t qfrag = base_u + C::OFF_QFRAG;
  float qshift_f = 1.f;
  if constexpr (KV8) {
    float* qmax = reinterpret_cast<float*>(base + C::OFF_QMAX);
    int shift = 0;
    if (std::is_same<T, __nv_bfloat16>::value) {
      float mx = 0.f;
      for (int i = tid; i < 16 * C::CPR; i += C::CT) {
        const int r = i / C::CPR, ch = i - (i / C::CPR) * C::CPR;
        uint32_t w[4];
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(sQ + swz<C::ROW_BYTES>(r, ch)));
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
      asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");
      float m = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) m = fmaxf(m, qmax[w]);
      if (m > 0.f) {
        const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xff) - 127;
        shift = max(-100, min(100, e - 14));
      }
    }
    qshift_f = exp2f(static_cast<float>(shift));
    const float qmul = exp2f(static_cast<float>(-shift));
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
                     : "r"(sQ + swz<C::ROW_BYTES>(gg + 8 * h, d >> 3) + off));
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
  }

  const int g8 = lane >> 2, c4 = lane & 3;
  const int rA = g8, rB = g8 + 8;
  const int ctx = L - q_len;
  const int pA = ctx + rA / G, pB = ctx + rB / G;
  const bool okA = rA < rows, okB = rB < rows;
  float slopeA = 0.f, slopeB = 0.f;
  if (p.alibi) {
    if (okA) slopeA = p.alibi[g * G + rA % G];
    if (okB) slopeB = p.alibi[g * G + rB % G];
  }
  const bool plain = (p.softcap <= 0.f) && (p.alibi == nullptr);
  // soft-cap without ALiBi: interior tiles need only the capped logit
  const bool capped = (p.softcap > 0.f) && (p.alibi == nullptr);
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
  const float qk_scale = p.scale * (p.k_scale ? *p.k_scale : 1.f) * qshift_f;
  const float vscale = p.v_scale ? *p.v_scale : 1.f;
  const float scale_log2 = qk_scale * kLog2e;
  // keys every row admits: tiles inside [full_lo, full_hi) skip the mask
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
  const int lm_mi = lane >> 3, lm_r = lane & 7;
  const int kw0 = warp * C::KW;                 // this warp's keys in a tile

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % STAGES;
    const uint32_t par = (it / STAGES) & 1;
    const int kt = kt0 + it * KT;
    if (!mbar_wait_lim(full_k(s), par, abort_flag,
                        p.err, p.wait_ns)) break;
    const uint32_t sK = tile_k(s), sV = tile_v(s);
    if (const unsigned bad = bad_boxes[s]) {
      // pages the table pointed outside the cache: zero keys and values
      for (int idx = lane; idx < C::KW * C::RCH; idx += 32) {
        const int r = kw0 + idx / C::RCH, ch = idx % C::RCH;
        if (!((bad >> (r / RB)) & 1u)) continue;
        asm volatile("st.shared.v4.u32 [%0], {%2, %2, %2, %2};\n"
                     "st.shared.v4.u32 [%1], {%2, %2, %2, %2};" ::"r"(
                         sK + kv_off<KT, D, RG>(r, ch)),
                     "r"(sV + kv_off<KT, D, RG>(r, ch)), "r"(0)
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
      // one ldmatrix.x4 of code bytes holds 4 / NKT k16 steps of all NKT
      // n8 tiles: matrix m covers n8 tile m % NKT of step grp * 4 / NKT +
      // m / NKT (16 code bytes = one k16 step)
      constexpr int KPG = 4 / C::NKT;
#pragma unroll
      for (int grp = 0; grp < (D / 16) / KPG; ++grp) {
        uint32_t r4[4];
        {
          const int nt = lm_mi % C::NKT, ks = grp * KPG + lm_mi / C::NKT;
          ldmatrix_x4(sK + kv_off<KT, D, RG>(kw0 + nt * 8 + lm_r, ks), r4[0],
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
          ldmatrix_x4(sK + kv_off<KT, D, RG>(r, ch), b0, b1, b2, b3);
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
        for (int e = 0; e < 4; ++e) sc[nt][e] = post * tanh_fast(sc[nt][e] * pre);
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
                        p.err, p.wait_ns)) break;
    if (kt + kw0 + C::KW > hi) {
      // rows of this warp at or past the loaded range: zero them, so that
      // P = 0 never meets NaN padding or a stale row
      const int r0 = max(hi - kt, kw0);
      for (int idx = lane; idx < (kw0 + C::KW - r0) * C::RCH; idx += 32) {
        const int r = r0 + idx / C::RCH, ch = idx % C::RCH;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                         sV + kv_off<KT, D, RG>(r, ch)),
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
        // V^T fragments straight from the code bytes: the 8-bit transposing
        // ldmatrix of a 16-key x 16-column block gives each lane four keys
        // of column g8 (d0) and of column g8 + 8 (d1); the row addresses
        // take the keys in the order 2c, 2c + 1, 2c + 8, 2c + 9 (c = 0 ..
        // 3), so a lane's four are the B fragment's k = 2 c4, 2 c4 + 1,
        // 2 c4 + 8, 2 c4 + 9.
        const int li = lane & 15;
        const int kr = kw0 + ks * 16 + 2 * (li >> 2) + (li & 1) +
                       ((li & 2) ? 8 : 0);
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {
          uint32_t d0, d1, b0, b1, b2, b3;
          ldmatrix_b8_trans(sV + kv_off<KT, D, RG>(kr, q), d0, d1);
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
          ldmatrix_x4_trans(sV + kv_off<KT, D, RG>(r, ch), b0, b1, b2, b3);
          mma_16816<T>(o[2 * dp], a, b0, b1);
          mma_16816<T>(o[2 * dp + 1], a, b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);

  // every consumer has finished with the ring: it becomes the combine buffer
  asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");
  if (*abort_flag) return;
  float* sm_ml = reinterpret_cast<float*>(base);            // [NCW][16][2]
  float* sm_o = sm_ml + NCW * 16 * 2;                       // [NCW][16][D]
  if (c4 == 0) {
    sm_ml[(warp * 16 + g8) * 2 + 0] = mA;
    sm_ml[(warp * 16 + g8) * 2 + 1] = lA;
    sm_ml[(warp * 16 + g8 + 8) * 2 + 0] = mB;
    sm_ml[(warp * 16 + g8 + 8) * 2 + 1] = lB;
  }
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    *reinterpret_cast<float2*>(sm_o + (warp * 16 + g8) * D + dn * 8 + 2 * c4) =
        make_float2(o[dn][0], o[dn][1]);
    *reinterpret_cast<float2*>(sm_o + (warp * 16 + g8 + 8) * D + dn * 8 +
                               2 * c4) = make_float2(o[dn][2], o[dn][3]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(C::CT) : "memory");

  const bool split = p.chunk > 0;
  T* __restrict__ OUT = static_cast<T*>(p.out);
  for (int i = tid; i < rows * (D / 4); i += C::CT) {
    const int rr = i / (D / 4), c = (i - rr * (D / 4)) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm_ml[(w * 16 + rr) * 2]);
    const float mb = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float f = ex2(sm_ml[(w * 16 + rr) * 2] - mb);
      lsum += f * sm_ml[(w * 16 + rr) * 2 + 1];
      const float4 v =
          *reinterpret_cast<const float4*>(sm_o + (w * 16 + rr) * D + c);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    const int tok = q0 + rr / G, h = g * G + rr % G;
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
      if (p.lse && c == 0)
        p.lse[static_cast<int64_t>(h) * p.total_q + tok] = lse;
    } else {
      float* dst = p.part_o +
                   ((static_cast<int64_t>(blockIdx.y) * p.part_rows +
                       part_row(p.part_tpr, b, q0, tok)) *
                        p.Hq + h) * D + c;
      *reinterpret_cast<float4*>(dst) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (c == 0)
        p.part_lse[(static_cast<int64_t>(blockIdx.y) * p.Hq + h) *
                       p.part_rows +
                   part_row(p.part_tpr, b, q0, tok)] = lse;
    }
  }
}

// The kernel.  As a programmatic dependent launch (p.pdl_done set: the
// launch may start while the grid before it in the stream still runs, once
// that grid's CTAs have all signalled), every CTA counts itself done in
// *p.pdl_done and the last one waits for the grid before to complete, so
// this grid ends after it and work queued after this grid sees both
// grids' results.  Without a preceding grid the wait returns at once.
template <typename T, int D, int NCW, int KT, int STAGES, bool RG, bool KV8>
__global__ void __launch_bounds__((NCW + 1) * 32)
decode_tma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  // a prefill launch queued after this one in the same call may start
  // before this grid ends (it writes other requests' rows)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  decode_tma_body<T, D, NCW, KT, STAGES, RG, KV8>(p, tm_k, tm_v);
  if (p.pdl_done && threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    if (atomicAdd(reinterpret_cast<unsigned*>(p.pdl_done), 1u) == total - 1) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      *p.pdl_done = 0;
    }
  }
}

#ifndef PKV_DTMA_D128_STAGES
#define PKV_DTMA_D128_STAGES 2
#endif
#ifndef PKV_DTMA_D256_STAGES
#define PKV_DTMA_D256_STAGES 2
#endif
#ifndef PKV_DTMA_FP8_STAGES
#define PKV_DTMA_FP8_STAGES 4
#endif
#ifndef PKV_DTMA_D64_STAGES
#define PKV_DTMA_D64_STAGES 4
#endif

template <typename T, int D, int NCW, int KT, int STAGES, bool RG,
          bool KV8 = false>
cudaError_t launch_cfg(const AttnParams& p, const CUtensorMap& mk,
                       const CUtensorMap& mv, dim3 grid,
                       cudaStream_t stream) {
  using C = Cfg<D, NCW, KT, STAGES, KV8>;
  auto kern = decode_tma_kernel<T, D, NCW, KT, STAGES, RG, KV8>;
  cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  note_launch();
  if (!p.pdl_done) {
    kern<<<grid, C::NT, C::SMEM, stream>>>(p, mk, mv);
    return cudaGetLastError();
  }
  // programmatic dependent launch: CTAs may start on the SMs the grid
  // before leaves free, once all of that grid's CTAs have signalled
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p, mk, mv);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const AttnParams& p, int D, bool rg,
                     const CUtensorMap& mk, const CUtensorMap& mv, dim3 grid,
                     cudaStream_t s) {
  // E4M3 cache (D = 128): one-byte codes in 128-column boxes, 4 stages of
  // 64 keys (the bytes in flight of the 16-bit kernel's 2 stages)
  if (p.kv_fp8)
    return D == 128 ? launch_cfg<T, 128, 4, 64, PKV_DTMA_FP8_STAGES, false,
                                 true>(p, mk, mv, grid, s)
                    : cudaErrorInvalidValue;
  // row-group boxes at D = 128 only: D = 64 has one column block (both
  // layouts are the same), and at D = 256 their addressing took the
  // consumers from 200 to 245 registers, one CTA per SM fewer
  switch (D) {
    case 64:
      return launch_cfg<T, 64, 4, 64, PKV_DTMA_D64_STAGES, false>(p, mk, mv,
                                                                  grid, s);
    case 128:
      return rg ? launch_cfg<T, 128, 4, 64, PKV_DTMA_D128_STAGES, true>(
                      p, mk, mv, grid, s)
                : launch_cfg<T, 128, 4, 64, PKV_DTMA_D128_STAGES, false>(
                      p, mk, mv, grid, s);
    case 256:
      return launch_cfg<T, 256, 2, 32, PKV_DTMA_D256_STAGES, false>(p, mk, mv,
                                                                    grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dtma

int decode_tma_tile_keys(int D) { return D == 256 ? 32 : 64; }

cudaError_t launch_decode_attn_tma(const AttnParams& a, int D, bool bf16,
                                   int grid_x, cudaStream_t stream) {
  AttnParams p = a;
  const int KT = decode_tma_tile_keys(D);
  int RB = 16;
  while (RB * 2 <= KT && p.BS % (RB * 2) == 0) RB *= 2;
  if (p.cu_k) RB = KT;    // non-paged: a box may start on any row
  p.rb = RB;
  p.kv_order_hnd = p.c_sh > p.c_sr ? 1 : 0;
  CUtensorMap mk, mv;
  if (p.kv_fp8) {
    // E4M3 codes: a row of D = 128 is one 128-byte box column
    if (D != 128 || p.cu_k ||
        !make_kv_map_ex(&mk, p.kc, 0, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                        p.c_sr, p.c_sh, RB, p.kv_order_hnd) ||
        !make_kv_map_ex(&mv, p.vc, 0, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                        p.c_sr, p.c_sh, RB, p.kv_order_hnd))
      return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(p.batch) * p.Hkv, grid_x, 1);
    return bf16 ? dtma::dispatch<__nv_bfloat16>(p, D, false, mk, mv, grid,
                                                stream)
                : dtma::dispatch<__half>(p, D, false, mk, mv, grid, stream);
  }
  // one row-group box per page and matrix where the view allows it (the
  // 4-D boxes take one per page and 64-column block)
  const bool rg =
      D == 128 && !p.cu_k &&
      make_kv_rg_map(&mk, p.kc, bf16, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                     p.c_sr, p.c_sh, RB, p.kv_order_hnd) &&
      make_kv_rg_map(&mv, p.vc, bf16, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                     p.c_sr, p.c_sh, RB, p.kv_order_hnd);
  if (!rg &&
      (!make_kv_map(&mk, p.kc, bf16, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                    p.c_sr, p.c_sh, RB, p.kv_order_hnd) ||
       !make_kv_map(&mv, p.vc, bf16, D, p.BS, p.Hkv, p.num_blocks, p.c_sb,
                    p.c_sr, p.c_sh, RB, p.kv_order_hnd)))
    return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(p.batch) * p.Hkv, grid_x, 1);
  return bf16 ? dtma::dispatch<__nv_bfloat16>(p, D, rg, mk, mv, grid, stream)
              : dtma::dispatch<__half>(p, D, rg, mk, mv, grid, stream);
}

}  // namespace pkv
