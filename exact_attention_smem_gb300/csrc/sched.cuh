// Longest-processing-time-first (LPT) work ordering for the persistent kernels
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling", Summary: a longest-processing-time-first tile scheduler for
// causal masking and variable sequence lengths).
//
// A work unit is (sequence, row block, head). Its cost is the number of inner
// blocks it walks: for the forward, KV blocks of 128 keys seen by a block of
// query rows; for the backward, query blocks seen by a block of keys. Units are
// listed in non-increasing cost (Graham's LPT list order); ties go by sequence,
// then row block, then head, so the query heads sharing one KV head sit next
// to each other and read the same K/V from L2 at about the same time.
//
// The persistent grid deals the list out in "snake" rounds: in round r the G
// CTAs take the next G units, in CTA order for even r and reversed for odd r,
// which evens out the per-CTA sums. Every role of a CTA runs its own Walker
// over the same list, so they agree on the unit sequence without
// communicating; seeking is amortised O(1) per unit because the list is walked
// group by group ((cost level, sequence) groups of consecutive row blocks).
//
// Host and device share this code; the host build backs the scheduler tests.
#pragma once
#include <cstdint>

namespace fa {

struct SchedSpec {
  const int* cu;   // packed boundaries (nseq + 1), nullptr for dense
  int nseq;        // sequences (dense: batch)
  int Sq, Sk;      // dense lengths
  int heads;       // units per (sequence, row block)
  int causal;
  int unit_rows;   // rows per unit: fwd query rows, bwd keys
  int inner;       // rows per inner block: fwd keys per KV block, bwd query rows per block
  int kind;        // 0 forward, 1 backward

  __host__ __device__ __forceinline__ void seq(int i, int& qs, int& ql, int& ks, int& kl) const {
    if (cu) {
      qs = cu[i];
      ql = cu[i + 1] - cu[i];
      ks = qs;
      kl = ql;
    } else {
      qs = i * Sq;
      ql = Sq;
      ks = i * Sk;
      kl = Sk;
    }
  }
  // Number of row blocks (units per head) of sequence i.
  __host__ __device__ __forceinline__ int nblocks(int ql, int kl) const {
    const int n = kind == 0 ? ql : kl;
    return (n + unit_rows - 1) / unit_rows;
  }
  // Inner blocks walked by row block m.
  __host__ __device__ __forceinline__ int cost(int m, int ql, int kl) const {
    if (kind == 0) {
      if (!causal) return (kl + inner - 1) / inner;
      int last = m * unit_rows + unit_rows;
      last = last < ql ? last : ql;                 // one past the last query row
      int kend = last + (kl - ql);                  // keys visible to that row
      kend = kend < kl ? kend : kl;
      return kend <= 0 ? 0 : (kend + inner - 1) / inner;
    }
    const int nq = (ql + inner - 1) / inner;
    if (!causal) return nq;
    int r0 = m * unit_rows - (kl - ql);             // first query row seeing key m*unit_rows
    r0 = r0 > 0 ? r0 : 0;
    if (r0 >= ql) return 0;
    return nq - r0 / inner;
  }
  __host__ __device__ __forceinline__ int max_cost() const {
    int mx = 0;
    for (int i = 0; i < nseq; ++i) {
      int qs, ql, ks, kl;
      seq(i, qs, ql, ks, kl);
      const int nb = nblocks(ql, kl);
      if (nb == 0) continue;
      const int c = cost(kind == 0 ? nb - 1 : 0, ql, kl);
      mx = c > mx ? c : mx;
    }
    return mx;
  }
  // Row blocks of sequence i whose cost equals c: [lo, hi). Costs are monotone
  // in m (non-decreasing forward, non-increasing backward).
  __host__ __device__ __forceinline__ void range(int c, int ql, int kl, int& lo, int& hi) const {
    const int nb = nblocks(ql, kl);
    // first m with "cost beyond c on the far side": forward cost >= c / backward cost <= c
    int a = 0, b = nb;
    while (a < b) {
      const int mid = (a + b) >> 1;
      const int cm = cost(mid, ql, kl);
      if (kind == 0 ? (cm >= c) : (cm <= c)) b = mid; else a = mid + 1;
    }
    lo = a;
    a = lo;
    b = nb;
    while (a < b) {
      const int mid = (a + b) >> 1;
      const int cm = cost(mid, ql, kl);
      if (kind == 0 ? (cm > c) : (cm < c)) b = mid; else a = mid + 1;
    }
    hi = a;
  }
};

struct Unit {
  int seq, m, head, cost;
  int q_start, q_len, k_start, k_len;
};

// Walks the LPT list: groups (cost level desc, sequence asc), inside a group row
// blocks ascending then heads.
struct Walker {
  SchedSpec s;
  int level, seq_i, lo, hi;      // current group
  long long gstart;              // list index of the group's first unit
  int qs, ql, ks, kl;
  bool done;

  __host__ __device__ __forceinline__ void init(const SchedSpec& spec) {
    s = spec;
    level = s.max_cost();
    seq_i = -1;
    gstart = 0;
    lo = hi = 0;
    done = false;
    advance_group();
  }
  __host__ __device__ __forceinline__ void advance_group() {
    gstart += (long long)(hi - lo) * s.heads;
    for (;;) {
      ++seq_i;
      if (seq_i >= s.nseq) {
        seq_i = 0;
        --level;
        if (level < 0) {
          done = true;
          lo = hi = 0;
          return;
        }
      }
      if (s.nseq == 0) {
        done = true;
        return;
      }
      s.seq(seq_i, qs, ql, ks, kl);
      if (s.nblocks(ql, kl) == 0) continue;
      s.range(level, ql, kl, lo, hi);
      if (hi > lo) return;
    }
  }
  // Position on list entry `target` (targets must not decrease between calls).
  __host__ __device__ __forceinline__ bool seek(long long target, Unit& u) {
    while (!done && target >= gstart + (long long)(hi - lo) * s.heads) advance_group();
    if (done) return false;
    const long long off = target - gstart;
    u.seq = seq_i;
    u.m = lo + (int)(off / s.heads);
    u.head = (int)(off % s.heads);
    u.cost = level;
    u.q_start = qs;
    u.q_len = ql;
    u.k_start = ks;
    u.k_len = kl;
    return true;
  }
};

// List index of the k-th unit of CTA b among G (snake rounds).
__host__ __device__ __forceinline__ long long snake_index(int k, int G, int b) {
  return (long long)k * G + ((k & 1) ? (G - 1 - b) : b);
}

}  // namespace fa
