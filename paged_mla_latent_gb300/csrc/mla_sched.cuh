// Split-KV work decomposition shared by the decode kernel (every warp role walks the
// same sequence) and the merge kernel (which finds the partials of each output).
//
// The history of every request is divided into pieces that run on different CTAs and
// are combined afterwards with softmax weights: the "history partitions" of
// "Scaling Kimi K3 on AMD Instinct MI355X" §4 "MLA" (work assigned to workgroups within
// one GPU, KV storage unchanged) and the normalised partials of §1 "Cache".
//
// Work unit u = (request b, row group g).  A request's T_b * H query rows (token-major,
// head-minor, as q is laid out) are cut into groups of NG rows; each group is one MMA
// N-tile and attends all L_b positions of its request.
//
// Two policies:
//  * auto (num_kv_splits <= 0): the units are laid end to end in a "global position"
//    line of length W = groups * (kv_indptr[B] - kv_indptr[0]) and CTA i of Gp takes
//    [floor(i W / Gp), floor((i+1) W / Gp)).  Every CTA gets the same number of cache
//    rows regardless of how lengths are distributed (batch 1 with a 142K history fills
//    every SM; 16 requests of 68K split ~10 ways each).  The piece of unit u on CTA i
//    writes partial slot i + u (unique: see unit_partials).  A unit lying on one CTA is
//    written directly, with no merge.
//  * fixed (num_kv_splits = k >= 1): unit u is cut into k equal pieces p = u*k + j,
//    CTA i runs pieces i, i + grid, ...; partial slot = p; k = 1 writes directly.
#pragma once

#include <stdint.h>

// Host + device when compiled by nvcc; plain host code otherwise (the CPU test-suite
// compiles this header with g++ to simulate the schedule).
#ifdef __CUDACC__
#define PMLA_HD __host__ __device__
#else
#define PMLA_HD
#endif

namespace pmla {

constexpr int kTile = 128;          // cache positions per pipeline tile (MMA M)
constexpr int kD = 576;             // latent entry width
constexpr int kDV = 512;            // value width
constexpr int kMinChunk = 256;      // auto policy: at least this many rows per CTA

// Rows per group (MMA N of the QK product) for a call with max_seqlen_q * H rows per
// request.  Fewer groups means fewer passes over the same cache rows.
PMLA_HD inline int pick_group_rows(int rows_per_request) {
  if (rows_per_request <= 16) return 16;
  if (rows_per_request <= 32) return 32;
  return 48;
}
PMLA_HD inline int groups_for(int rows_per_request, int ng) {
  return (rows_per_request + ng - 1) / ng;
}

struct SchedParams {
  const int32_t* kv_indptr;
  const int32_t* qo_indptr;
  int B;
  int H;
  int NG;
  int groups;      // row groups per request
  int splits;      // <= 0 auto, else fixed pieces per unit
  int grid;        // CTAs launched
};

struct Piece {
  int b, g;        // request, row group
  int j0, j1;      // positions [j0, j1) of the request
  int L, T;        // request kv_len and q_len
  int rows;        // real query rows in this group (<= NG)
  int64_t slot;    // partial slot (ignored when direct)
  bool direct;     // this piece is the whole unit: write o / lse directly
  int64_t kv0;     // kv_indptr[b]: position j of the request is kv_indices[kv0 + j]
  int qo0;         // qo_indptr[b]: first query token of the request
};

// Effective CTA count of the auto policy for a line of W positions.
PMLA_HD inline int auto_ctas(int64_t W, int grid) {
  int64_t g = W / kMinChunk;
  if (g < 1) g = 1;
  if (g > grid) g = grid;
  return static_cast<int>(g);
}

// CTA of the auto policy that owns global position x (0 <= x < W).
PMLA_HD inline int auto_cta_of(int64_t x, int64_t W, int Gp) {
  return static_cast<int>(((x + 1) * Gp - 1) / W);
}

// Largest b in [0, B) with groups * (kv_indptr[b] - kv_indptr[0]) <= x.
PMLA_HD inline int find_request(const int32_t* kvp, int B, int groups, int64_t x) {
  const int32_t kv0 = kvp[0];
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(groups) * (kvp[mid] - kv0) <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Positions [j0, j1) of piece k of a unit with L positions under the fixed policy.
PMLA_HD inline void piece_bounds(int L, int splits, int k, int* j0, int* j1) {
  *j0 = static_cast<int>(static_cast<int64_t>(k) * L / splits);
  *j1 = static_cast<int>(static_cast<int64_t>(k + 1) * L / splits);
}

// Iterator over one CTA's pieces.  Every role of a CTA constructs it with the same
// arguments and so sees the same sequence.  Pieces without work (no real rows, no
// positions) are skipped.  On inconsistent indptr data it stops and sets *bad.
struct PieceIter {
  SchedParams sp;
  int cta;
  int64_t W;
  int Gp;
  int64_t x, x1;       // auto policy cursor
  int64_t p, p_end;    // fixed policy cursor
  Piece held;          // returned again by the next call of next() when have_held
  bool have_held;

  // Every member is assigned on every path: the iterator is only ever constructed with
  // init(), never copied.
  PMLA_HD void init(const SchedParams& s, int cta_id) {
    sp.kv_indptr = s.kv_indptr;
    sp.qo_indptr = s.qo_indptr;
    sp.B = s.B;
    sp.H = s.H;
    sp.NG = s.NG;
    sp.groups = s.groups;
    sp.splits = s.splits;
    sp.grid = s.grid;
    cta = cta_id;
    W = 0;
    Gp = 0;
    x = x1 = 0;
    p = p_end = 0;
    have_held = false;
    held = Piece{0, 0, 0, 0, 0, 0, 0, 0, false, 0, 0};
    if (sp.splits <= 0) {
      W = static_cast<int64_t>(sp.groups) * (sp.kv_indptr[sp.B] - sp.kv_indptr[0]);
      Gp = auto_ctas(W, sp.grid);
      if (W <= 0 || cta >= Gp) {
        x = x1 = 0;
      } else {
        x = W * cta / Gp;
        x1 = W * (cta + 1) / Gp;
      }
    } else {
      p = cta;
      p_end = static_cast<int64_t>(sp.B) * sp.groups * sp.splits;
    }
  }

  // Make the next call of next() return pc again (the piece it returned last), so that a
  // piece computed once up front is not recomputed from memory by every role.
  PMLA_HD void hold(const Piece& pc) {
    held = pc;
    have_held = true;
  }

  PMLA_HD bool next(Piece& pc, int* bad) {
    if (have_held) {
      have_held = false;
      pc = held;
      return true;
    }
    while (true) {
      if (sp.splits <= 0) {
        if (x >= x1) return false;
        const int b = find_request(sp.kv_indptr, sp.B, sp.groups, x);
        const int64_t base = static_cast<int64_t>(sp.groups) * (sp.kv_indptr[b] - sp.kv_indptr[0]);
        const int L = sp.kv_indptr[b + 1] - sp.kv_indptr[b];
        const int64_t off = x - base;
        if (L <= 0 || off < 0 || off >= static_cast<int64_t>(L) * sp.groups) {
          *bad = 1;
          x = x1;
          return false;
        }
        const int g = static_cast<int>(off / L);
        const int j0 = static_cast<int>(off - static_cast<int64_t>(g) * L);
        const int64_t room = x1 - x;
        const int j1 = (L - j0 <= room) ? L : j0 + static_cast<int>(room);
        x += j1 - j0;
        pc.b = b;
        pc.g = g;
        pc.j0 = j0;
        pc.j1 = j1;
        pc.L = L;
        pc.slot = static_cast<int64_t>(cta) + static_cast<int64_t>(b) * sp.groups + g;
        pc.direct = (j0 == 0 && j1 == L);
      } else {
        if (p >= p_end) return false;
        const int64_t u = p / sp.splits;
        const int k = static_cast<int>(p - u * sp.splits);
        const int b = static_cast<int>(u / sp.groups);
        const int g = static_cast<int>(u - static_cast<int64_t>(b) * sp.groups);
        const int L = sp.kv_indptr[b + 1] - sp.kv_indptr[b];
        if (L < 0) {
          *bad = 1;
          p = p_end;
          return false;
        }
        pc.b = b;
        pc.g = g;
        piece_bounds(L, sp.splits, k, &pc.j0, &pc.j1);
        pc.L = L;
        pc.slot = p;
        pc.direct = (sp.splits == 1);
        p += sp.grid;
      }
      pc.kv0 = sp.kv_indptr[pc.b];
      pc.qo0 = sp.qo_indptr[pc.b];
      pc.T = sp.qo_indptr[pc.b + 1] - pc.qo0;
      const int rows_req = pc.T * sp.H;
      int rows = rows_req - pc.g * sp.NG;
      if (rows > sp.NG) rows = sp.NG;
      pc.rows = rows;
      if (rows > 0 && pc.j1 > pc.j0) return true;
    }
  }
};

// Number of partial slots a call needs (host and device agree on this bound).
PMLA_HD inline int64_t partial_slots(int B, int groups, int splits, int grid) {
  const int64_t units = static_cast<int64_t>(B) * groups;
  if (splits <= 0) return units + grid;
  if (splits == 1) return 0;
  return units * splits;
}

// Partials of unit (b, g) as the decode kernel wrote them: slots first .. first+count-1
// (fixed policy: some may be empty pieces, see piece_bounds).  Returns false when the
// unit needs no merge: it ran whole on one CTA (written directly) or has no positions.
PMLA_HD inline bool unit_partials(const SchedParams& sp, int b, int g, int64_t* first,
                                  int* count) {
  const int L = sp.kv_indptr[b + 1] - sp.kv_indptr[b];
  if (L <= 0) return false;
  const int64_t u = static_cast<int64_t>(b) * sp.groups + g;
  if (sp.splits <= 0) {
    const int64_t W = static_cast<int64_t>(sp.groups) * (sp.kv_indptr[sp.B] - sp.kv_indptr[0]);
    const int Gp = auto_ctas(W, sp.grid);
    const int64_t xs = static_cast<int64_t>(sp.groups) * (sp.kv_indptr[b] - sp.kv_indptr[0]) +
                       static_cast<int64_t>(g) * L;
    const int i0 = auto_cta_of(xs, W, Gp);
    const int i1 = auto_cta_of(xs + L - 1, W, Gp);
    if (i0 == i1) return false;
    *first = static_cast<int64_t>(i0) + u;   // CTA i writes unit u's piece to slot i + u
    *count = i1 - i0 + 1;
    return true;
  }
  if (sp.splits == 1) return false;
  *first = u * sp.splits;
  *count = sp.splits;
  return true;
}

}  // namespace pmla
