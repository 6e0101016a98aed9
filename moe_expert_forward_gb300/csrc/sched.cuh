// Tile-group scheduling shared by the persistent GEMM kernels.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace mm {

constexpr int kQueue = 8;                  // tile groups the scheduler may run ahead of a CTA's roles
constexpr int kSiteQueueFull = 107;        // default wait site of a queue read

struct Task {
  int type;      // 1 = L1, 2 = L2
  int e, n, b, valid;
  bool last;     // the last pool block of its tile group
  bool rev;      // walk the contraction from its last k-block down (odd blocks of a group)
};

// Tasks are dealt to the persistent CTAs in tile groups: one weight tile (e, n)
// of one GEMM together with every pool block of expert e.  A CTA takes a
// group's blocks back to back, so the second and later blocks of an expert
// find the tile's weights still in L2 instead of reading them from HBM again.
// Every other block walks the contraction backwards: it starts with the
// k-blocks its predecessor loaded last, the ones most likely still in L2 when
// the 152 CTAs' tiles together are larger than L2.
// Group order: modes 1/2, expert-major then tile; mode 3, segment u = expert
// u's NB1 L1 groups followed by expert (u - lag)'s NB2 L2 groups.  The number
// of groups per segment does not depend on the routing, so a group index
// decodes in closed form; groups of experts without tokens are skipped.
struct Cursor {
  int i = 0;            // next queue position
  int bl = 0, nb = 0;   // block within the current group, blocks of its expert
  Task t;
};

// Tile groups taken by this CTA, in order: slot i % kQueue holds the i-th
// (-1 once there are none left).  The scheduler thread fills a slot after
// every consumer has released it.
struct Queue {
  uint64_t* full;       // [kQueue], one arrival: the slot holds a group
  uint64_t* empty;      // [kQueue], kQueueConsumers arrivals: the slot is free
  volatile int* g;      // [kQueue]
};

struct Sched {
  const int* blk;   // [E+1] pool-block offsets per expert
  const int* cnt;   // [E]
  int E, NB1, NB2, mode, lag;
  int BT = kBT;     // pool rows per block
  // false: a group is one weight tile with every pool block of its expert, taken
  // back to back by one CTA; true: a group is one (weight tile, pool block) pair,
  // so the blocks of one tile are dealt to neighbouring free CTAs, which stream
  // the tile's k-blocks at about the same time (the second read hits L2)
  bool per_block = false;

  __device__ __forceinline__ int largest_leq(const int* a, int n, int v, int scale) const {
    int lo = 0, hi = n - 1;                  // largest i < n with a[i] * scale <= v
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a[mid] * scale <= v) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
  // units of expert-range [0, u): experts (tile groups) or pool blocks (per block)
  __device__ __forceinline__ int units(int u) const { return per_block ? blk[u] : u; }
  __device__ __forceinline__ int groups() const {
    return mode == 1 ? units(E) * NB1 : (mode == 2 ? units(E) * NB2 : units(E) * (NB1 + NB2));
  }
  // mode 3: groups in the segments before segment u
  __device__ __forceinline__ int groups_before(int u) const {
    const int l1 = u < E ? u : E;
    int l2 = u - lag;
    l2 = l2 < 0 ? 0 : (l2 > E ? E : l2);
    return units(l1) * NB1 + units(l2) * NB2;
  }
  // Group g's task (expert, tile, type); *bl receives its pool block within the
  // expert when groups are per block (0 otherwise).
  __device__ __forceinline__ void group(int g, Task& t, int* bl) const {
    int u, r;
    if (mode != 3) {
      const int nbw = mode == 1 ? NB1 : NB2;
      t.type = mode;
      u = per_block ? largest_leq(blk, E, g, nbw) : g / nbw;
      r = g - units(u) * nbw;
    } else {
      int lo = 0, hi = E + lag - 1;            // the segment holding group g
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (groups_before(mid) <= g) lo = mid; else hi = mid - 1;
      }
      u = lo;
      r = g - groups_before(lo);
      const int n1 = lo < E ? NB1 * (per_block ? blk[lo + 1] - blk[lo] : 1) : 0;
      if (r < n1) {
        t.type = 1;
      } else {
        t.type = 2;
        u = lo - lag;
        r -= n1;
      }
    }
    t.e = u;
    if (per_block) {
      const int nb = blk[u + 1] - blk[u];
      t.n = r / nb;
      *bl = r - t.n * nb;
    } else {
      t.n = r;
      *bl = 0;
    }
  }
  __device__ __forceinline__ void block(Cursor& c) const {
    c.t.b = blk[c.t.e] + c.bl;
    const int rem = cnt[c.t.e] - c.bl * BT;
    c.t.valid = rem < BT ? rem : BT;
    if (per_block) {
      // the expert's other blocks of this tile run concurrently on other CTAs:
      // keep the weights in L2 unless this is the tile's only reader
      c.t.last = blk[c.t.e + 1] - blk[c.t.e] == 1;
      c.t.rev = false;
    } else {
      c.t.last = c.bl + 1 == c.nb;
      c.t.rev = (c.bl & 1) != 0;
    }
  }
  __device__ __forceinline__ int group_blocks(int g) const {
    if (per_block) return 1;                   // every per-block group has its block
    Task t;
    int bl;
    group(g, t, &bl);
    return blk[t.e + 1] - blk[t.e];
  }
  // Advance to this CTA's next task; false when there is none (or on abort).
  // A warp-wide consumer calls this with all 32 lanes converged: lane 0 takes
  // the queue slot and broadcasts it.
  __device__ __forceinline__ bool next(Cursor& c, const Queue& q, const Status& st, volatile int* abort,
                                       bool warp_wide, int lane, int site = kSiteQueueFull) const {
    if (c.bl + 1 < c.nb) {
      ++c.bl;
      block(c);
      return true;
    }
    const int slot = c.i % kQueue;
    const uint32_t parity = (c.i / kQueue) & 1;
    ++c.i;
    int g = -1;
    if (!warp_wide || lane == 0) {
      if (mbar_wait(&q.full[slot], parity, st, abort, site)) {
        g = q.g[slot];
        mbar_arrive(&q.empty[slot]);
      }
    }
    if (warp_wide) g = __shfl_sync(0xffffffffu, g, 0);
    c.nb = 0;
    if (g < 0) return false;
    int bl;
    group(g, c.t, &bl);
    if (per_block) {
      c.bl = bl;
      c.nb = bl + 1;                           // this group's only block
    } else {
      c.nb = blk[c.t.e + 1] - blk[c.t.e];
      c.bl = 0;
    }
    block(c);
    return true;
  }
};


// The scheduler thread of a CTA.  Tile groups are taken from one counter shared
// by all CTAs, in increasing order, so CTAs that are free start neighbouring
// groups at about the same time: an expert's token block is read by its tiles
// while it is still in L2, and no CTA is left with a longer tail of static
// work.  Groups of experts without tokens are skipped here.
__device__ __forceinline__ void run_scheduler(const Sched& sch, const Queue& q, int* counter, const Status& st,
                                              volatile int* abort, int site) {
  const int ng = sch.groups();
  for (int i = 0;; ++i) {
    const int slot = i % kQueue;
    if (!mbar_wait(&q.empty[slot], ((i / kQueue) & 1) ^ 1, st, abort, site)) break;
    int g = -1;
    for (;;) {
      const int x = atomicAdd(counter, 1);
      if (x >= ng) break;
      if (sch.group_blocks(x) > 0) {
        g = x;
        break;
      }
    }
    q.g[slot] = g;
    mbar_arrive(&q.full[slot]);
    if (g < 0) break;
  }
}

}  // namespace mm
