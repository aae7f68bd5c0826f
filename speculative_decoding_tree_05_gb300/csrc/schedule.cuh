// schedule.cuh -- key-range groups: the units (request, row tile, key range)
// that a CTA pair of the prefix pass computes when a batch is divided by key
// ranges instead of by fixed-length splits.
//
// The requests' 64-key steps are laid end to end, request 0 first: K steps in
// all, request b's at [off(b), off(b) + steps(b)).  The pairs form G groups of
// row_tiles pairs (G <= K: see groups_used); group g takes steps
// [floor(gK/G), floor((g+1)K/G)) and its
// pair t computes row tile t over them, one unit per request that the range
// touches.  So every group has the same number of steps however the lengths
// are mixed, a pair runs one unit more than there are request boundaries in
// its range, and the pairs of a group read the same keys at about the same
// time (the rows stay in L2 for the other tiles).  Piece k of request b is
// the part computed by group owner(off(b)) + k; its partial result goes to
// split slot k of the request, and the merge takes pieces(b) slots.
#pragma once
#include <cstdint>
#include "kernels.cuh"

namespace ddt {

// Groups in use: with fewer steps than groups (K < G) only the first K groups
// get a range (one step each), so that no range is empty and a request's
// pieces come from consecutive groups.
__host__ __device__ inline int groups_used(int G, int64_t K) { return K < G ? static_cast<int>(K) : G; }

// first step of group g (of G groups in use)
__host__ __device__ inline int64_t group_begin(int g, int64_t K, int G) { return int64_t(g) * K / G; }

// the group whose steps hold step x, 0 <= x < K: the largest g with
// floor(gK/G) <= x, i.e. with gK <= (x+1)G - 1
__host__ __device__ inline int group_owner(int64_t x, int64_t K, int G) {
  return static_cast<int>(((x + 1) * G - 1) / K);
}

// number of groups (pieces) that a request with steps [off, off + n) spans, G
// the groups launched
__host__ __device__ inline int group_pieces(int64_t off, int64_t n, int64_t K, int G) {
  G = groups_used(G, K);
  return n <= 0 ? 0 : group_owner(off + n - 1, K, G) - group_owner(off, K, G) + 1;
}

// The idx-th unit (0-based, in request order) of group g, G the groups
// launched: its request *b, keys [*kbegin, *kend) and piece number; false once
// the group has no more units.
// off(r), steps(r), keys(r): request r's first step, its number of steps and
// its number of keys.  Every argument is the same in all threads.
#pragma nv_exec_check_disable
template <class Off, class Steps, class Keys>
__host__ __device__ inline bool nth_group_unit(int g, int G, int64_t K, int batch, int idx, Off off, Steps steps,
                                               Keys keys, int* b, int* kbegin, int* kend, int* piece) {
  G = groups_used(G, K);
  if (g >= G) return false;
  const int64_t lo = group_begin(g, K, G), hi = group_begin(g + 1, K, G);
  int seen = 0;
  for (int r = 0; lo < hi && r < batch; ++r) {
    const int64_t o = off(r), n = steps(r);
    if (o >= hi) break;
    if (n == 0 || o + n <= lo) continue;
    if (seen++ < idx) continue;
    const int64_t s0 = lo > o ? lo : o, s1 = hi < o + n ? hi : o + n;
    const int64_t ke = (s1 - o) * kKeysPerTile;
    const int L = keys(r);
    *b = r;
    *kbegin = static_cast<int>((s0 - o) * kKeysPerTile);
    *kend = static_cast<int>(ke < L ? ke : L);
    *piece = g - group_owner(o, K, G);
    return true;
  }
  return false;
}

// The requests' steps as seen by one warp (batch <= 64: lane l holds requests
// l and l + 32).  Lengths outside [0, max_len] are clamped as everywhere else
// and flagged in `bad`; a null prefix_len means every request has max_len keys.
// Every lane of the warp must call it and the accessors, with the same b.
struct StepTable {
  int64_t first[2];  // first step of requests lane, lane + 32
  int32_t n[2];      // their steps
  int32_t len[2];    // their keys
  int64_t total;     // K
  bool bad;          // some request's length was out of range

  __device__ int64_t off(int b) const { return __shfl_sync(0xffffffffu, b < 32 ? first[0] : first[1], b & 31); }
  __device__ int64_t steps(int b) const { return __shfl_sync(0xffffffffu, b < 32 ? n[0] : n[1], b & 31); }
  __device__ int keys(int b) const { return __shfl_sync(0xffffffffu, b < 32 ? len[0] : len[1], b & 31); }
};

__device__ inline StepTable step_table(const int32_t* prefix_len, int max_len, int batch, int lane) {
  StepTable t;
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = lane + 32 * h;
    int L = 0;
    if (b < batch) {
      L = prefix_len != nullptr ? __ldg(prefix_len + b) : max_len;
      if (L < 0 || L > max_len) {
        bad = true;
        L = L < 0 ? 0 : max_len;
      }
    }
    t.len[h] = L;
    t.n[h] = (L + kKeysPerTile - 1) / kKeysPerTile;
  }
  // inclusive running sums over the lanes, then the second half after the first
  int64_t s0 = t.n[0], s1 = t.n[1];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u0 = __shfl_up_sync(0xffffffffu, s0, o), u1 = __shfl_up_sync(0xffffffffu, s1, o);
    if (lane >= o) {
      s0 += u0;
      s1 += u1;
    }
  }
  s1 += __shfl_sync(0xffffffffu, s0, 31);
  t.first[0] = s0 - t.n[0];
  t.first[1] = s1 - t.n[1];
  t.total = __shfl_sync(0xffffffffu, s1, 31);
  t.bad = __any_sync(0xffffffffu, bad);
  return t;
}

}  // namespace ddt
