// mbarrier and TMA helpers shared by the kernels that move K/V pages with
// the tensor-memory accelerator (cp.async.bulk.tensor), and the host-side
// tensor-map builder for a paged cache view.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "pkv_common.cuh"

namespace pkv {

constexpr uint32_t kSpinLimit = 1u << 28;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled
// column block whose rows are 128 bytes apart (the layout a TMA box with
// CU_TENSOR_MAP_SWIZZLE_128B and a 128-byte inner extent writes).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false when the CTA is aborting, or after limit_ns (then
// the error word gets kErrTimeout and the CTA-wide abort flag is raised).
__device__ __forceinline__ bool mbar_wait_lim(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag,
                                              unsigned* err,
                                              uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    // the time is read after the second poll (a limit of 0 gives up there)
    // and then every 256 polls
    if (it == 1 || (it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 >= limit_ns || it > kSpinLimit) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          unsigned* err) {
  return mbar_wait_lim(bar, parity, abort_flag, err, kWaitLimitNs);
}

// Wait used while draining in-flight work: no abort check, still bounded.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (mbar_try(bar, parity)) return;
    if ((it & 255u) == 255u && globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap,
                                            int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(bar)
      : "memory");
}

// L2 cache policy for data read exactly once: its lines are the first
// candidates for eviction, so they do not push out lines that are re-read.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  return pol;
}

// tma_load_4d with an L2 cache policy (l2_evict_first_policy).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst,
                                                 const void* tmap, int c0,
                                                 int c1, int c2, int c3,
                                                 uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], "
      "%7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* tmap,
                                            int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

// tma_load_5d with an L2 cache policy (l2_evict_first_policy).
__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst,
                                                 const void* tmap, int c0,
                                                 int c1, int c2, int c3,
                                                 int c4, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], "
      "[%7], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap,
                                            int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
      "r"(bar)
      : "memory");
}

// Tiled TMA store of a 3-D box from shared memory (bulk-group completion;
// the box's inner coordinate c0 must be a multiple of 16 bytes).
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src,
                                             int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group "
      "[%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Every committed bulk store has finished reading its shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed bulk store is complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Bounded wait until *cnt >= target, for a count that only grows: false
// when the CTA is aborting, or after kWaitLimitNs (then the error word gets
// kErrTimeout and the CTA-wide abort flag is raised).
__device__ __forceinline__ bool count_wait(const volatile int* cnt,
                                           int target,
                                           volatile int* abort_flag,
                                           unsigned* err) {
  if (*cnt >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (*cnt >= target) return true;
    if (it == 1 || (it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 >= kWaitLimitNs || it > kSpinLimit) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D map over one cache view [NB, BS, Hkv, D] (element strides s_blk,
// s_row, s_head; unit stride along D): dims (D, Hkv, BS, NB) for NHD
// strides, (D, BS, Hkv, NB) when the head stride is the larger (HND).  The
// box is 64 x 1 x RB x 1 (NHD) or 64 x RB x 1 x 1 (HND) elements, 128-byte
// swizzled.  False if the driver entry point is missing or rejects the map.
bool make_kv_map(CUtensorMap* map, const void* ptr, bool bf16, int D, int BS,
                 int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                 int64_t s_head, int RB, bool hnd);
// Row-group map of a 16-bit cache view: one box of RB keys (RB a multiple
// of 8, at most block_size) holds every 64-column block of one page and
// lands as [8-key group][column block][8 keys][64 columns]; coordinates
// (0, 0, 0, page * (BS / 8) + row / 8, head) for NHD views and (0, 0, 0,
// row / 8, page * Hkv + head) for HND views.  False when the view's
// strides do not allow it (NHD needs s_blk = BS s_row, HND s_blk = Hkv
// s_head).
bool make_kv_rg_map(CUtensorMap* map, const void* ptr, bool bf16, int D,
                    int BS, int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                    int64_t s_head, int RB, bool hnd);
// The same map for an element type `elem`: 0 = one-byte codes (E4M3; box
// 128 x 1 x RB x 1), 1 = f16, 2 = bf16 (box 64 x 1 x RB x 1).  Strides are
// in elements of that type.
bool make_kv_map_ex(CUtensorMap* map, const void* ptr, int elem, int D,
                    int BS, int Hkv, int64_t NB, int64_t s_blk, int64_t s_row,
                    int64_t s_head, int RB, bool hnd);

}  // namespace pkv
