// Longest-processing-time-first (LPT) work ordering for the persistent kernels
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling", Summary: a longest-processing-time-first tile scheduler for
// causal masking and variable sequence lengths).
//
// A work unit is (sequence, row block, head). Its cost is the number of inner
// blocks it walks: for the forward, KV blocks of 128 keys seen by a block of
// query rows; for the backward, query blocks seen by a block of keys.
//
// The list is cut into head groups (`hblock` consecutive heads, all sequences)
// processed one after the other; inside a group units are listed in
// non-increasing cost (Graham's LPT list order), ties by sequence, row block,
// then head. Grouping keeps the data the concurrently running CTAs share —
// K/V of the forward, the fp32 dQ accumulator and Q/dO of the backward — small
// enough to stay in L2 (the host picks `hblock` so that one group holds at
// least one unit per CTA); LPT inside each group keeps the long units first,
// and since groups follow each other without a barrier, only the last group's
// short tail limits the balance at the end.
//
// The persistent grid deals the list out in "snake" rounds: in round r the G
// CTAs take the next G units, in CTA order for even r and reversed for odd r,
// which evens out the per-CTA sums. Every role of a CTA runs its own Walker
// over the same list, so they agree on the unit sequence without
// communicating. Dense layouts seek directly (O(log) per unit, seek_dense);
// packed layouts walk the list group by group ((cost level, sequence) groups
// of consecutive row blocks): every CTA passes every (level, sequence) pair
// once, at two cost evaluations for a pair outside the sequence's cost range
// (a few hundred sequences cost well under a millisecond).
//
// Host and device share this code; the host build backs the scheduler tests.
#pragma once
#include <cstdint>

namespace fa {

// x / d for x >= 0; a shift when d is a power of two (it always is here: 64,
// 128 or 256 rows), so the scheduler's arithmetic stays off the divide path.
__host__ __device__ __forceinline__ int div_nonneg(int x, int d) {
  if ((d & (d - 1)) == 0) {
    int sh = 0;
    while ((1 << sh) < d) ++sh;
    return x >> sh;
  }
  return x / d;
}

struct SchedSpec {
  const int* cu;   // packed boundaries (nseq + 1), nullptr for dense
  int nseq;        // sequences (dense: batch)
  int Sq, Sk;      // dense lengths
  int heads;       // units per (sequence, row block)
  int causal;
  int unit_rows;   // rows per unit: fwd query rows, bwd keys
  int inner;       // rows per inner block: fwd keys per KV block, bwd query rows per block
  int kind;        // 0 forward, 1 backward
  int hblock;      // heads per group (>= 1)
  const int* cu_k = nullptr;  // packed key boundaries when they differ from cu, or
  int k_off = 0;              // else at cu[k_off + i] (0: the query boundaries)

  __host__ __device__ __forceinline__ void seq(int i, int& qs, int& ql, int& ks, int& kl) const {
    if (cu) {
      qs = cu[i];
      ql = cu[i + 1] - cu[i];
      if (cu_k) {
        ks = cu_k[i];
        kl = cu_k[i + 1] - cu_k[i];
      } else {
        ks = cu[k_off + i];
        kl = cu[k_off + i + 1] - ks;
      }
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
    return div_nonneg(n + unit_rows - 1, unit_rows);
  }
  // Inner blocks walked by row block m.
  __host__ __device__ __forceinline__ int cost(int m, int ql, int kl) const {
    if (kind == 0) {
      if (!causal) return div_nonneg(kl + inner - 1, inner);
      int last = m * unit_rows + unit_rows;
      last = last < ql ? last : ql;                 // one past the last query row
      int kend = last + (kl - ql);                  // keys visible to that row
      kend = kend < kl ? kend : kl;
      return kend <= 0 ? 0 : div_nonneg(kend + inner - 1, inner);
    }
    const int nq = div_nonneg(ql + inner - 1, inner);
    if (!causal) return nq;
    int r0 = m * unit_rows - (kl - ql);             // first query row seeing key m*unit_rows
    r0 = r0 > 0 ? r0 : 0;
    if (r0 >= ql) return 0;
    return nq - div_nonneg(r0, inner);
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

// Walks the list: head groups in order; inside a group (cost level desc,
// sequence asc) groups of units, inside those row blocks ascending then heads.
struct Walker {
  SchedSpec s;
  int maxc, hb, h0, hcount;      // current head group: heads [h0, h0 + hcount)
  int level, seq_i, lo, hi;      // current (level, sequence) run
  long long gstart;              // list index of the run's first unit
  int qs, ql, ks, kl;
  bool done;

  __host__ __device__ __forceinline__ void set_hblock(int b) {
    hb = b;
    h0 = b * s.hblock;
    const int left = s.heads - h0;
    hcount = left < s.hblock ? left : s.hblock;
  }
  __host__ __device__ __forceinline__ void init(const SchedSpec& spec) {
    s = spec;
    if (s.hblock < 1) s.hblock = 1;
    maxc = s.max_cost();
    set_hblock(0);
    level = maxc;
    seq_i = -1;
    gstart = 0;
    lo = hi = 0;
    done = s.nseq == 0 || s.heads <= 0;
    if (!done) advance_group();
  }
  __host__ __device__ __forceinline__ void advance_group() {
    gstart += (long long)(hi - lo) * hcount;
    lo = hi = 0;
    for (;;) {
      ++seq_i;
      if (seq_i >= s.nseq) {
        seq_i = 0;
        --level;
        if (level < 0) {
          if (h0 + hcount >= s.heads) {
            done = true;
            return;
          }
          set_hblock(hb + 1);
          level = maxc;
        }
      }
      s.seq(seq_i, qs, ql, ks, kl);
      const int nb = s.nblocks(ql, kl);
      if (nb == 0) continue;
      // costs are monotone in the block index: the end blocks bound this
      // sequence's levels, so most (level, sequence) pairs skip the searches
      const int c0 = s.cost(0, ql, kl), c1 = s.cost(nb - 1, ql, kl);
      if (level < (c0 < c1 ? c0 : c1) || level > (c0 < c1 ? c1 : c0)) continue;
      s.range(level, ql, kl, lo, hi);
      if (hi > lo) return;
    }
  }
  // Dense layouts (every sequence has the same lengths): the entry at any list
  // index follows directly. Inside a head group the list holds, per row block
  // in order of decreasing cost, nseq x hcount units; so the p-th block in that
  // order (m = p for the backward, whose cost falls with m; m = nb-1-p for the
  // forward, whose cost grows with m) fixes the cost level, and the level's
  // block range fixes sequence, block and head. O(log nb) per call instead of
  // a walk over every group before the target.
  __host__ __device__ __forceinline__ bool seek_dense(long long target, Unit& u) const {
    int qs0, ql, ks0, kl;
    s.seq(0, qs0, ql, ks0, kl);
    const int nb = s.nblocks(ql, kl);
    if (nb == 0 || s.nseq <= 0 || s.heads <= 0 || target < 0) return false;
    const long long per_head = (long long)nb * s.nseq;
    const long long full = per_head * s.hblock;
    const long long hg = target / full;
    if (hg * s.hblock >= s.heads) return false;
    const int h0g = (int)(hg * s.hblock);
    const int hc = s.heads - h0g < s.hblock ? s.heads - h0g : s.hblock;
    const long long o = target - hg * full;
    if (o >= per_head * hc) return false;
    const long long per_block = (long long)s.nseq * hc;
    const int pos = (int)(o / per_block);
    const int mp = s.kind == 0 ? nb - 1 - pos : pos;
    const int c = s.cost(mp, ql, kl);
    int rlo, rhi;
    s.range(c, ql, kl, rlo, rhi);
    const long long r = o - (long long)(s.kind == 0 ? nb - rhi : rlo) * per_block;
    const long long per_seq = (long long)(rhi - rlo) * hc;
    const int sq = (int)(r / per_seq);
    const long long rem = r - (long long)sq * per_seq;
    u.seq = sq;
    u.m = rlo + (int)(rem / hc);
    u.head = h0g + (int)(rem % hc);
    u.cost = c;
    s.seq(sq, u.q_start, u.q_len, u.k_start, u.k_len);
    return true;
  }

  // Position on list entry `target` (targets must not decrease between calls).
  __host__ __device__ __forceinline__ bool seek(long long target, Unit& u) {
    if (s.cu == nullptr) return seek_dense(target, u);
    while (!done && target >= gstart + (long long)(hi - lo) * hcount) advance_group();
    if (done) return false;
    const long long off = target - gstart;
    u.seq = seq_i;
    u.m = lo + (int)(off / hcount);
    u.head = h0 + (int)(off % hcount);
    u.cost = level;
    u.q_start = qs;
    u.q_len = ql;
    u.k_start = ks;
    u.k_len = kl;
    return true;
  }
};

// Heads per group: the fewest heads whose units cover `grid` CTAs at least once.
__host__ __device__ __forceinline__ int pick_hblock(long long units_per_head, int heads, int grid) {
  if (units_per_head <= 0) return heads > 0 ? heads : 1;
  long long hb = (grid + units_per_head - 1) / units_per_head;
  if (hb < 1) hb = 1;
  if (hb > heads) hb = heads;
  return (int)hb;
}

// List index of the k-th unit of CTA b among G (snake rounds).
__host__ __device__ __forceinline__ long long snake_index(int k, int G, int b) {
  return (long long)k * G + ((k & 1) ? (G - 1 - b) : b);
}

}  // namespace fa
