// Distribution of a scheduler work list over the persistent CTAs of the tensor-core
// kernels.
//
// The list is sorted heavy-first.  Handing item it, it + grid, it + 2 grid, ... to CTA
// `it` fixes each CTA's share before the kernel starts; the CTAs then finish up to 6%
// apart (their items differ slightly, and so do their SMs' speeds), and the kernel lasts
// as long as the slowest.  Instead, each CTA can take its next item from a counter in
// the workspace header when it is ready for one: the heaviest items go first and the
// last ones are the lightest, so the CTAs finish within about one light item of each
// other.  The assignment then changes from run to run, the results do not: every item
// is computed by one CTA alone, in the same order of operations.
//
// In a CTA, one thread (the claimer: the producer that loads each item's first tile)
// takes the index, loads the item and publishes it in a ring of kFeedSlots slots in
// shared memory, with a FULL barrier per slot (one arrival) and an EMPTY barrier per
// slot (one arrival per reading role).  Every other role reads the items from the ring
// in order.  A role whose warp runs two cursors over the items (an issuer one step
// ahead of itself) reads each slot twice and arrives from the lagging cursor only.
//
// Claiming costs the claimer an atomic and a list load per item, about a thousand
// cycles under load, which is small against an item of many steps and not against one
// of one or two.  The scheduler therefore decides per list: it sets the counter to 0
// (claimed) when the items average enough steps, and to -1 (fixed assignment)
// otherwise.  With DYN = false the assignment is always fixed and the feed compiles to
// the per-role list walk alone (the softmax kernels, whose workloads' items are short,
// and the rotary kernels, whose compute warps look ahead in the list).
#pragma once

#include "internal.h"
#include "tc_ptx.cuh"

namespace jfa {
namespace tc {

// The slowest reader (an issuer of an item's last products) trails the claimer by
// about two items of a few steps each; with fewer slots the claimer would wait for it.
constexpr int kFeedSlots = 8;

// Shared-memory addresses of one CTA's feed ring: FULL[s] at bar0 + 8 s, EMPTY[s] at
// bar0 + 8 (kFeedSlots + s), slot s (one WorkItem; cost < 0 ends the list) at
// slot0 + 32 s.
struct FeedRing {
  uint32_t bar0, slot0;
};

__device__ __forceinline__ void st_shared_item(uint32_t a, const WorkItem& x) {
  asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x.b), "r"(x.h), "r"(x.tile),
               "r"(x.cost)
               : "memory");
  asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16), "r"(x.q0), "r"(x.k0), "r"(x.lq),
               "r"(x.lk)
               : "memory");
}
__device__ __forceinline__ WorkItem ld_shared_item(uint32_t a) {
  WorkItem x;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.b), "=r"(x.h), "=r"(x.tile), "=r"(x.cost)
               : "r"(a)
               : "memory");
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.q0), "=r"(x.k0), "=r"(x.lq), "=r"(x.lk)
               : "r"(a + 16)
               : "memory");
  return x;
}

// A reader's cursor over the CTA's items.
template <bool DYN>
struct Feed {
  FeedRing ring;
  uint32_t k;    // items taken (claimed mode)
  bool dyn;      // claimed mode
  const WorkItem* list;
  int n_items;
  int it;        // next list index (fixed assignment)
  WorkItem nxt;  // the item at `it`, loaded one item ahead (fixed assignment)

  __device__ void init(const FeedRing& r, const WorkItem* l, const int* ctr, int n) {
    ring = r;
    list = l;
    n_items = n;
    k = 0;
    it = blockIdx.x;
    // -1 (fixed assignment) stays -1; in claimed mode the counter is >= 0 throughout
    // the launch, including after the rewind at its end
    dyn = DYN && *reinterpret_cast<const volatile int*>(ctr) >= 0;
    if (!dyn && it < n_items) nxt = load_item(list, it);
  }

  // Fixed assignment: the next item of this CTA, or false at the end.
  __device__ bool next_fixed(WorkItem& w) {
    if (it >= n_items) return false;
    w = nxt;
    it += gridDim.x;
    if (it < n_items) nxt = load_item(list, it);
    return true;
  }

  // The next item: the fixed one, or in the claimer's order; false at the end of the
  // list or when a bounded wait gave up.  `warp_wide`: the whole warp runs this role's
  // loop (lane 0 arrives once every lane has read the slot); otherwise one thread does.
  // `arrive`: this cursor is the role's last reader of each slot.
  __device__ bool take(WorkItem& w, bool warp_wide, bool arrive, volatile int* abort, int* status) {
    if (!dyn) return next_fixed(w);
    const uint32_t s = k % kFeedSlots;
    if (!mbar_wait(ring.bar0 + 8u * s, (k / kFeedSlots) & 1u, abort, status)) return false;
    const WorkItem x = ld_shared_item(ring.slot0 + 32u * s);
    if (arrive) {
      if (warp_wide) __syncwarp();
      if (!warp_wide || (threadIdx.x & 31) == 0) mbar_arrive(ring.bar0 + 8u * (kFeedSlots + s));
    }
    ++k;
    if (x.cost < 0) return false;
    w = x;
    return true;
  }
};

// The claimer (one thread).  Each call returns the CTA's next item, false at the end of
// the list or when a bounded wait gave up (then nothing more is published; the other
// roles see the abort flag).  Items are published one ahead of what the claimer
// returns, so that the other producer can load the next item's tiles while this one
// still loads the current item's, and indices are taken two ahead, so that neither the
// counter's round trip nor the list load is waited for where it is issued: the index
// taken at one call is loaded at the next and published at the one after.
//
// Every claimer stops at the first index past the end, so each CTA takes exactly one
// such index, as its last: they are n_items, n_items + 1, ..., n_items + grid - 1.  The
// CTA that takes the last of them is the last to touch the counter in the launch and
// sets it back to 0, so that the next launch over the same list (a list reused by
// several calls) starts from the beginning.  A CTA that gives up in a bounded wait
// stops claiming early; the counter then stays where it is, and the lists must be
// built again (the status word reports the timeout).
template <bool DYN>
struct FeedClaimer {
  Feed<DYN> f;   // fixed assignment, ring and published count
  int* counter;
  int idx;       // the index taken last
  WorkItem cur;  // the item published last, returned by the next call
  WorkItem nxt;  // the item loaded last, published by the next call
  bool nxt_end;  // nxt is the end of the list

  __device__ void init(const FeedRing& r, const WorkItem* l, int* ctr, int n) {
    f.init(r, l, ctr, n);
    counter = ctr;
  }
  __device__ int take_index() {
    const int i = atomicAdd(counter, 1);
    if ((long long)i == (long long)f.n_items + gridDim.x - 1) atomicExch(counter, 0);
    return i;
  }
  __device__ bool publish(const WorkItem& x, volatile int* abort, int* status) {
    const uint32_t s = f.k % kFeedSlots;
    if (!mbar_wait(f.ring.bar0 + 8u * (kFeedSlots + s), ((f.k / kFeedSlots) & 1u) ^ 1u, abort, status))
      return false;
    st_shared_item(f.ring.slot0 + 32u * s, x);
    mbar_arrive(f.ring.bar0 + 8u * s);
    ++f.k;
    return true;
  }
  // Starts loading list item i into nxt (or marks the end).  The loads write nxt's
  // registers directly and are volatile, so that they are waited for only where nxt is
  // read, a whole item later.
  __device__ void fetch(int i) {
    nxt_end = (unsigned)i >= (unsigned)f.n_items;
    if (nxt_end) return;
    const int4* q = reinterpret_cast<const int4*>(f.list + i);
    asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(nxt.b), "=r"(nxt.h), "=r"(nxt.tile), "=r"(nxt.cost)
                 : "l"(q));
    asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(nxt.q0), "=r"(nxt.k0), "=r"(nxt.lq), "=r"(nxt.lk)
                 : "l"(q + 1));
  }
  __device__ bool claim(WorkItem& w, volatile int* abort, int* status) {
    if (!f.dyn) return f.next_fixed(w);
    if (f.k == 0) {  // prime: item 0 published, item 1 loading, item 2's index taken
      WorkItem x0{};
      x0.cost = -1;
      const int i0 = f.n_items > 0 ? take_index() : f.n_items;
      if ((unsigned)i0 < (unsigned)f.n_items) x0 = load_item(f.list, i0);
      cur = x0;
      if (!publish(cur, abort, status)) return false;
      if (cur.cost < 0) {
        nxt_end = true;
      } else {
        fetch(take_index());
        if (!nxt_end) idx = take_index();
      }
    }
    const WorkItem x = cur;  // published at the previous call
    if (x.cost < 0) return false;
    WorkItem y = nxt;  // loaded at the previous call: the item after x (or the end)
    if (nxt_end) y.cost = -1;
    if (!publish(y, abort, status)) return false;
    cur = y;
    if (!nxt_end) {
      fetch(idx);  // taken at the previous call
      if (!nxt_end) idx = take_index();
    }
    w = x;
    return true;
  }
};

}  // namespace tc
}  // namespace jfa
