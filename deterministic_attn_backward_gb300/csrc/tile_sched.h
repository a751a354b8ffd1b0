// tile_sched.h -- tile schedules of the deterministic attention backward.
//
// One definition, evaluated by the main kernel on the device and by the host
// introspection / DAG-simulator functions.  Pure integer arithmetic.
//
// Terms (DASH, "Deterministic Attention Scheduling for High-throughput
// Reproducible LLM Training", technical summary section 2):
//   N        number of 128-row tiles of a head (S / 128), for KV and for Q.
//   chain    all steps of one KV tile, run back to back on one CTA so that dK
//            and dV accumulate on chip (section 2.1, constraint).
//   unit     what one CTA takes at a time: one chain, or for the causal
//            symmetric shift a pair of chains (KV p, then KV N-1-p).
//   rank     rank(i, j) = position of KV tile i in dQ_j's fixed reduction
//            order (section 1: a fixed accumulation order for dQ).
#pragma once

#if defined(__CUDACC__)
#define DAB_HD __host__ __device__ __forceinline__
#else
#define DAB_HD inline
#endif

namespace dab {

enum : int { kSchedSerial = 0, kSchedDescending = 1, kSchedShift = 2, kSchedAtomic = 3 };
enum : int { kMaskFull = 0, kMaskCausal = 1 };

// Full-mask shift: the cyclic walk needs every KV tile of a gang co-resident.
// Heads with more than kShiftGroup tiles are split into groups of kShiftGroup
// consecutive KV tiles; dQ_j is reduced group by group, and inside a group in
// visit order.  A constant (not the SM count), so the bits do not depend on
// the grid.
constexpr int kShiftGroup = 128;

struct Step {
  int kv;            // KV tile i
  int q;             // Q tile j
  bool chain_first;  // first step of a chain: dK/dV accumulators start at 0
  bool chain_last;   // last step of a chain: dK/dV are written out after it
};

DAB_HD int units_per_head(int sched, int mask, int N) {
  return (sched == kSchedShift && mask == kMaskCausal) ? N / 2 : N;
}

DAB_HD int unit_steps(int sched, int mask, int N, int u) {
  if (mask == kMaskFull) return N;
  if (sched == kSchedShift) return N + 1;  // chain p (N - p steps) + chain N-1-p (p + 1)
  return N - u;                            // causal chain of KV tile u: Q tiles u..N-1
}

// Step t of unit u.
DAB_HD Step step(int sched, int mask, int N, int u, int t) {
  Step s;
  if (sched == kSchedShift && mask == kMaskCausal) {
    // Symmetric shift (DASH summary sec. 2.2.B, causal): CTA p owns KV tiles p
    // and N-1-p.  Phase 1 (dense lower-left square): KV p against Q tiles
    // M..N-1, cyclically offset by p.  Phase 2 (folded triangles): M+1
    // positions, position x < M standing for Q tile x of KV p (upper-left
    // triangle) or Q tile N-2-x of KV N-1-p, position M for Q tile N-1; CTA p
    // visits positions p, p+1, ... (mod M+1), which finishes KV p's chain and
    // then walks KV N-1-p's Q tiles from N-1 down to N-1-p.
    const int M = N / 2, p = u;
    if (t < M) {
      s.kv = p;
      s.q = M + (p + t) % M;
      s.chain_first = (t == 0);
      s.chain_last = false;
      return s;
    }
    const int tp = t - M;              // 0..M
    const int pos = (p + tp) % (M + 1);
    if (tp < M - p) {                  // rest of KV p's chain: Q tiles p..M-1
      s.kv = p;
      s.q = pos;
      s.chain_first = false;
      s.chain_last = (tp == M - p - 1);
    } else {                           // KV N-1-p: Q tiles N-1, N-2, ..., N-1-p
      s.kv = N - 1 - p;
      s.q = (pos == M) ? N - 1 : N - 2 - pos;
      s.chain_first = (tp == M - p);
      s.chain_last = (tp == M);
    }
    return s;
  }
  const int steps = unit_steps(sched, mask, N, u);
  s.kv = u;
  s.chain_first = (t == 0);
  s.chain_last = (t == steps - 1);
  if (sched == kSchedShift) {                 // full mask: i, i+1, ..., i-1
    s.q = (u + t) % N;
  } else if (sched == kSchedDescending) {     // N-1 down to 0 (or down to i)
    s.q = N - 1 - t;
  } else {                                    // serial / atomic: ascending
    s.q = (mask == kMaskCausal) ? u + t : t;
  }
  return s;
}

DAB_HD int contributors(int mask, int N, int j) { return mask == kMaskCausal ? j + 1 : N; }

DAB_HD bool visible(int mask, int i, int j) { return mask == kMaskFull || j >= i; }

// rank(i, j); -1 for a masked tile or an unordered (atomic) schedule.
DAB_HD int rank(int sched, int mask, int N, int i, int j) {
  if (!visible(mask, i, j) || sched == kSchedAtomic) return -1;
  if (sched == kSchedSerial || sched == kSchedDescending) return i;  // ascending KV
  if (mask == kMaskCausal) {
    // Symmetric shift: visit order (see step()).  Q tiles j >= M get the M
    // phase-1 contributions first, in cyclic order (j - M - i) mod M, then the
    // phase-2 ones of KV tiles M..j in ascending i.  Q tiles j < M only get
    // phase-2 contributions, KV j first and KV 0 last.
    const int M = N / 2;
    if (j >= M) return (i < M) ? ((j - M - i) % M + M) % M : i;
    return j - i;
  }
  // Full-mask shift: group-major, then visit order inside the group.  KV tile
  // i visits Q tile j at step s_i = (j - i) mod N.
  const int g = i / kShiftGroup;
  const int a = g * kShiftGroup;
  const int L = (N - a < kShiftGroup) ? N - a : kShiftGroup;
  const int si = ((j - i) % N + N) % N;
  const int s0 = ((j - a) % N + N) % N;  // step of the group's first tile (the largest s)
  int pos;
  if (s0 - (L - 1) >= 0) {
    pos = si - (s0 - (L - 1));           // steps s0-L+1 .. s0, no wrap
  } else if (si <= s0) {
    pos = si;                            // wrapped: steps 0..s0 come first
  } else {
    pos = (s0 + 1) + (si - (N - (L - 1 - s0)));
  }
  return a + pos;
}

// Units that must be resident at the same time (the cyclic wait of shift).
DAB_HD int gang_size(int sched, int mask, int N) {
  if (sched != kSchedShift) return 1;
  if (mask == kMaskCausal) return N / 2;
  return N < kShiftGroup ? N : kShiftGroup;
}

// Shift units are placed statically (unit U on CTA U mod grid, in ascending
// U), which keeps every gang co-resident; the other schedules take units from
// a global counter in ascending order, which balances unequal causal chains.
DAB_HD bool static_dispatch(int sched) { return sched == kSchedShift; }

}  // namespace dab
