// Stream-K work split shared by the persistent expert kernels: every CTA takes an
// equal (or cost-weighted) contiguous share of all units' pipeline steps, and
// walks the (unit, step range) segments of its share in one fixed order that all
// of its roles agree on.
#pragma once
#include <cstdint>

#include "layout.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// Bounded wait that ignores the abort flag: used at teardown to let copies and
// MMAs already in flight land before shared and tensor memory are released.
// (8e8 SM cycles: about 0.4 s.)
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long c0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - c0 > 800000000ll) return;
  }
}

// Bounded wait until the n counters at p (raised by other CTAs of the grid with
// a fence then an atomic add) all reach `target`; then this thread's later bulk
// copies see the data written before those releases. Gives up like mbar_wait.
__device__ __noinline__ bool wait_counters(const int32_t* p, int n, int target, volatile int* abort_flag,
                                           int* status, uint32_t limit_kcycles) {
  const long long c0 = clock64();
  for (;;) {
    int below = 0;
    for (int k = 0; k < n; ++k) below += ld_relaxed_gpu(p + k) < target ? 1 : 0;
    if (below == 0) break;
    if (*abort_flag) return false;
    if (((clock64() - c0) >> 10) > static_cast<long long>(limit_kcycles)) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
    __nanosleep(256);
  }
  __threadfence();             // acquire: pairs with the writers' fence before their add
  fence_proxy_async_global();  // and orders the bulk copies (async proxy) after it
  return true;
}

struct Sched {
  long long W;           // total steps
  int G;                 // CTAs
  const long long* tab;  // [G + 1] cost-weighted first steps (shared memory), or null: even split
  int gran;              // even split: shares start at multiples of gran (W is a multiple)
  __device__ __forceinline__ long long start(int c) const {
    return tab ? tab[c] : gran * (static_cast<long long>(c) * (W / gran) / G);
  }
  // CTA whose share contains step g.
  __device__ int cta_of(long long g) const {
    if (tab) {  // the last CTA whose share starts at or before g
      int lo = 0, hi = G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab[mid] <= g)
          lo = mid;
        else
          hi = mid - 1;
      }
      return lo;
    }
    int c = static_cast<int>((g * G) / (W > 0 ? W : 1));
    if (c > G - 1) c = G - 1;
    while (c + 1 < G && start(c + 1) <= g) ++c;
    while (c > 0 && start(c) > g) --c;
    return c;
  }
};

// The segments (unit, step range) of a CTA's share [begin, end): a share starts
// and ends inside units that other CTAs share. Those partial units come first
// (the one the share starts in, then the one it ends in), then the whole units in
// order: every contributor to a split unit then reaches it early in its share, so
// the split unit's cross-CTA reduction (partial sums, ticket, last arriver)
// overlaps the whole units that follow instead of adding to the kernel's tail.
// Every role walks the same sequence.
struct SegIter {
  long long g, gend;  // the share
  long long uw;       // next whole unit (stage 2)
  int KBn;
  int stage;          // 0: first partial unit, 1: last partial unit, 2: whole units
  __device__ SegIter(long long begin, long long end, int kbn)
      : g(begin), gend(end), uw(0), KBn(kbn), stage(0) {}
  __device__ __forceinline__ void range(long long u, int& kb0, int& kb1) const {
    const long long lo = g - u * KBn, hi = gend - u * KBn;
    kb0 = static_cast<int>(lo > 0 ? lo : 0);
    kb1 = static_cast<int>(hi < KBn ? hi : KBn);
  }
  // Next (unit, step range) of this CTA's share.
  __device__ __forceinline__ bool next(long long& u, int& kb0, int& kb1) {
    if (gend <= g) return false;
    const long long u0 = g / KBn, u1 = (gend - 1) / KBn;
    const bool p0 = g > u0 * KBn || gend < (u0 + 1) * KBn;  // the share starts inside u0 (or ends in it)
    const bool p1 = u1 != u0 && gend < (u1 + 1) * KBn;       // the share ends inside u1
    if (stage == 0) {
      stage = 1;
      uw = p0 ? u0 + 1 : u0;
      if (p0) {
        u = u0;
        range(u, kb0, kb1);
        return true;
      }
    }
    if (stage == 1) {
      stage = 2;
      if (p1) {
        u = u1;
        range(u, kb0, kb1);
        return true;
      }
    }
    if (uw > (p1 ? u1 - 1 : u1)) return false;
    u = uw++;
    range(u, kb0, kb1);
    return true;
  }
};

}  // namespace
}  // namespace moe
