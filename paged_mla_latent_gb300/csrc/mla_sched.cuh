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
//  * auto (num_kv_splits <= 0): the units are laid end to end on a cost line and CTA i of
//    Gp takes [floor(i W / Gp), floor((i+1) W / Gp)) of its length W.  Each (unit, row
//    group) occupies e + w L: a fixed cost e for the piece's set-up and epilogue, then w
//    per position.  Every CTA thus gets the same estimated time regardless of how
//    lengths are distributed (batch 1 with a 142K history fills every SM; 16 requests of
//    68K split ~10 ways each), and a CTA whose range crosses into another unit gets fewer
//    positions for the extra piece.  The piece of unit u on CTA i writes partial slot
//    i + u (unique: see unit_partials).  A unit lying on one CTA is written directly,
//    with no merge.
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

// Rows per group for a call with max_seqlen_q * H rows per request: 16, 32 or 48 (the
// kernel with positions on the tensor-memory lanes, rows on the MMA's N), or 96 (the kernel
// with the rows on the lanes) for more than 48.  Fewer groups means fewer passes over the
// same cache rows.
PMLA_HD inline int pick_group_rows(int rows_per_request) {
  if (rows_per_request <= 16) return 16;
  if (rows_per_request <= 32) return 32;
  if (rows_per_request <= 48) return 48;
  return 96;
}
PMLA_HD inline int groups_for(int rows_per_request, int ng) {
  return (rows_per_request + ng - 1) / ng;
}

// What a schedule covers.  kSchedWhole: every request's positions, as described above.
// kSchedCascade serves a batch whose requests share their first P cache positions (the
// prefix-cache pattern of the captured concurrency-16/24 workloads: "[Kimi-K3 MLA TP8]
// MLA performance" §1 "Environment" and §5.4).  Its line holds two kinds of units:
//  * v < VP: prefix units.  Unit v is a group of gsize consecutive requests attending
//    positions [0, P) together.  Their query rows are consecutive in q (request-major), so
//    a group is one MMA N-tile and each shared cache row is read once per group instead of
//    once per request.  No causal masking: every query of the group sees the whole prefix.
//  * v = VP + b: request b attending its own positions [P, L_b).
// Every unit writes partials; the cascade merge combines each row's prefix and own parts.
// P comes from the caller, who knows its prefix cache (mla_decode_shared_prefix);
// prefixes shorter than kMinShared are not split off.
// kSchedCascadePaged is the cascade on pages of several tokens: the same schedule, in its
// own kernel instantiation, so that the one-token-page cascade carries no page arithmetic
// (with it, the c16 cascade call took 2 us longer).
enum : int { kSchedWhole = 0, kSchedCascade = 1, kSchedCascadePaged = 2 };
constexpr int kMinShared = 1024;
// The schedule functions take the mode as a template argument: a compile-time mode gives
// the decode kernel only its own code path (the plain decode carries none of the cascade's
// arithmetic); kSchedAny reads it from SchedParams::mode (merge kernels, host tests).
constexpr int kSchedAny = -1;

struct SchedParams {
  const int32_t* kv_indptr;
  const int32_t* qo_indptr;
  int B;
  int H;
  int NG;
  int groups;      // row groups per (virtual) request
  int splits;      // <= 0 auto, else fixed pieces per unit
  int grid;        // CTAs launched
  int mode;        // kSchedWhole / kSchedCascade
  int gsize;       // kSchedCascade: requests per prefix unit
  int shared;      // kSchedCascade: the shared prefix length P
  // Cost line of the auto policy (0 reads as 1, as w_own, as 0 respectively):
  int w_own;       // per position of a request's (own) positions
  int w_prefix;    // kSchedCascade: per position of a prefix unit
  int piece_cost;  // per (unit, row group): set-up and epilogue of a piece
  // Paged caches: kv_indptr counts pages of 2^log2_page tokens and the last page of request
  // b holds last_page_lens[b] of them (0 / null: one token a page).  kSchedCascade: the
  // shared prefix P is a whole number of pages.
  int log2_page;
  const int32_t* last_page_lens;
};

// Cost-line weights the library sets.  A piece's fixed cost (its epilogue, the pipeline's
// refill) is charged as 512 positions: a sweep of 192 .. 768 on every workload put the
// optimum at 512 to 768.  Prefix and own units take the same weight per position: with one
// softmax warpgroup per 16 query rows a 48-row prefix tile costs what a 12-row own tile
// does (cheaper prefix weights measured slower).
// The cascade in 96-row groups (mla_decode_rows96.cuh) charges 256 positions a piece and a
// prefix position 1.15 own positions: its 12-row own pieces end with a short epilogue, its
// 96-row prefix pieces with a long one (~6.4 us), and its prefix tiles carry the full
// softmax.  A sweep of 128 .. 512 positions and 1.0 .. 1.35 put the optimum there (c16
// shared prefix 59.9 -> 56.4 us, c24 74.6 -> 71.7 us, the 128-token-page cascade within
// 0.5 %).
constexpr int kPieceCostPositions = 512;
constexpr int kCascade96PieceCost = 256;
constexpr int kCascade96OwnWeight = 20;      // prefix : own = 23 : 20 = 1.15
constexpr int kCascade96PrefixWeight = 23;
inline void sched_set_costs(SchedParams* sp, int /*rows_per_request*/) {
  if (sp->mode != kSchedWhole && sp->NG == 96) {
    sp->w_own = kCascade96OwnWeight;
    sp->w_prefix = kCascade96PrefixWeight;
    sp->piece_cost = kCascade96PieceCost * kCascade96OwnWeight;
    return;
  }
  sp->w_own = 1;
  sp->w_prefix = 0;   // reads as w_own
  sp->piece_cost = kPieceCostPositions;
}

struct Piece {
  int b, g;        // (virtual) request, row group
  int j0, j1;      // positions [j0, j1) of the (virtual) request
  int L, T;        // its kv_len and query tokens
  int cfrom;       // causal masking applies to positions > cfrom + (token index)
  int rows;        // real query rows in this group (<= NG)
  int64_t slot;    // partial slot (ignored when direct)
  bool direct;     // this piece is the whole unit: write o / lse directly
  int64_t kv0;     // position j of the piece's request is kv_indices[kv0 + j]
  int qo0;         // first query token of the (virtual) request
};

template <int MODE>
PMLA_HD inline int sched_mode(const SchedParams& sp) {
  const int m = MODE == kSchedAny ? sp.mode : MODE;
  return m == kSchedCascadePaged ? kSchedCascade : m;
}
// log2 of the tokens a page: 0 at compile time for the one-token-page cascade.
template <int MODE>
PMLA_HD inline int sched_lg(const SchedParams& sp) {
  return MODE == kSchedCascade ? 0 : sp.log2_page;
}

// The shared prefix length a schedule uses (0 in whole mode or below kMinShared).
template <int MODE = kSchedAny>
PMLA_HD inline int64_t sched_shared(const SchedParams& sp) {
  if (sched_mode<MODE>(sp) == kSchedWhole) return 0;
  const int64_t P = sp.shared;
  return P >= kMinShared ? P : 0;
}

// Prefix units of a cascade schedule.
PMLA_HD inline int sched_prefix_units(const SchedParams& sp) {
  return (sp.B + sp.gsize - 1) / sp.gsize;
}

// Number of units on the line (per row group).
template <int MODE = kSchedAny>
PMLA_HD inline int sched_requests(const SchedParams& sp) {
  return sched_mode<MODE>(sp) == kSchedCascade ? sched_prefix_units(sp) + sp.B : sp.B;
}

// Cache positions of all units before v (per row group), and of v itself.
template <int MODE = kSchedAny>
PMLA_HD inline int64_t sched_cum(const SchedParams& sp, int64_t P, int v) {
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    if (v <= VP) return static_cast<int64_t>(v) * P;
    const int b = v - VP;
    return static_cast<int64_t>(VP) * P +
           (static_cast<int64_t>(sp.kv_indptr[b]) - sp.kv_indptr[0]) * (int64_t{1} << sched_lg<MODE>(sp)) -
           static_cast<int64_t>(b) * P;
  }
  return (static_cast<int64_t>(sp.kv_indptr[v]) - sp.kv_indptr[0]) * (int64_t{1} << sched_lg<MODE>(sp));
}
template <int MODE = kSchedAny>
PMLA_HD inline int sched_len(const SchedParams& sp, int64_t P, int v) {
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    if (v < VP) return static_cast<int>(P);
    return (sp.kv_indptr[v - VP + 1] - sp.kv_indptr[v - VP]) * (1 << sched_lg<MODE>(sp)) -
           static_cast<int>(P);
  }
  return (sp.kv_indptr[v + 1] - sp.kv_indptr[v]) * (1 << sched_lg<MODE>(sp));
}
// Positions unit v really holds: its page-rounded length (sched_len) less the unused slots
// of its request's last page (a prefix unit's P positions are whole pages).  The schedule
// line is laid out in page-rounded lengths (prefix sums of kv_indptr); pieces and merge
// ranges are clipped to this.
template <int MODE = kSchedAny>
PMLA_HD inline int sched_real_len(const SchedParams& sp, int64_t P, int v) {
  const int L = sched_len<MODE>(sp, P, v);
  if (sched_lg<MODE>(sp) == 0 || L <= 0 || !sp.last_page_lens) return L;
  int b = v;
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    if (v < VP) return L;
    b = v - VP;
  }
  const int ps = 1 << sched_lg<MODE>(sp);
  int last = sp.last_page_lens[b];
  last = last < 1 ? 1 : (last > ps ? ps : last);   // out of range: flagged by mla_validate
  return L - ps + last;
}
// Tokens request b holds (its pages' slots less the unused ones of its last page).
template <int MODE = kSchedAny>
PMLA_HD inline int sched_req_len(const SchedParams& sp, int b) {
  const int pages = sp.kv_indptr[b + 1] - sp.kv_indptr[b];
  const int ps = 1 << sched_lg<MODE>(sp);
  if (ps == 1 || pages <= 0 || !sp.last_page_lens) return pages * ps;
  int last = sp.last_page_lens[b];
  last = last < 1 ? 1 : (last > ps ? ps : last);
  return (pages - 1) * ps + last;
}
// Cost-line weights of unit v and the fixed cost of a (unit, row group).
PMLA_HD inline int64_t sched_w_own(const SchedParams& sp) {
  return sp.w_own > 0 ? sp.w_own : 1;
}
template <int MODE = kSchedAny>
PMLA_HD inline int64_t sched_weight(const SchedParams& sp, int v) {
  if (sched_mode<MODE>(sp) == kSchedCascade && v < sched_prefix_units(sp))
    return sp.w_prefix > 0 ? sp.w_prefix : sched_w_own(sp);
  return sched_w_own(sp);
}
PMLA_HD inline int64_t sched_piece_cost(const SchedParams& sp) {
  return sp.piece_cost > 0 ? sp.piece_cost : 0;
}
// Cost-line start of unit v (per row group): the units before it, each e + w L.
template <int MODE = kSchedAny>
PMLA_HD inline int64_t sched_line(const SchedParams& sp, int64_t P, int v) {
  const int64_t e = sched_piece_cost(sp);
  const int64_t wo = sched_w_own(sp);
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    const int64_t unit_p = e + sched_weight<MODE>(sp, 0) * P;
    if (v <= VP) return static_cast<int64_t>(v) * unit_p;
    const int b = v - VP;
    return static_cast<int64_t>(VP) * unit_p + static_cast<int64_t>(b) * e +
           wo * ((static_cast<int64_t>(sp.kv_indptr[b]) - sp.kv_indptr[0]) *
                     (int64_t{1} << sched_lg<MODE>(sp)) -
                 static_cast<int64_t>(b) * P);
  }
  return static_cast<int64_t>(v) * e +
         wo * ((static_cast<int64_t>(sp.kv_indptr[v]) - sp.kv_indptr[0]) *
               (int64_t{1} << sched_lg<MODE>(sp)));
}
// Positions [0, L) of a (unit, row group) whose line segment starts d before line point
// x: position j sits at line point e + w j of the segment; returns how many positions lie
// before x.
PMLA_HD inline int line_positions(int64_t d, int64_t e, int64_t w, int L) {
  if (d <= e) return 0;
  const int64_t n = (d - e + w - 1) / w;
  return n < L ? static_cast<int>(n) : L;
}

// First index-array entry, query tokens [qo0, qo1) and causal base of unit v.
template <int MODE = kSchedAny>
PMLA_HD inline int64_t sched_kv0(const SchedParams& sp, int64_t P, int v) {
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    if (v < VP) return sp.kv_indptr[v * sp.gsize];
    return static_cast<int64_t>(sp.kv_indptr[v - VP]) + (P >> sched_lg<MODE>(sp));   // P: whole pages
  }
  return sp.kv_indptr[v];
}
template <int MODE = kSchedAny>
PMLA_HD inline void sched_tokens(const SchedParams& sp, int v, int* qo0, int* qo1) {
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    if (v < VP) {
      const int last = (v + 1) * sp.gsize < sp.B ? (v + 1) * sp.gsize : sp.B;
      *qo0 = sp.qo_indptr[v * sp.gsize];
      *qo1 = sp.qo_indptr[last];
      return;
    }
    v -= VP;
  }
  *qo0 = sp.qo_indptr[v];
  *qo1 = sp.qo_indptr[v + 1];
}
// Positions beyond cfrom + (token index) need the causal test; prefix units have none.
template <int MODE = kSchedAny>
PMLA_HD inline int sched_cfrom(const SchedParams& sp, int v, int L, int T) {
  if (sched_mode<MODE>(sp) == kSchedCascade && v < sched_prefix_units(sp)) return L;
  return L - T;
}

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

// Largest v in [0, VB) with groups * line(v) <= x.
template <int MODE = kSchedAny>
PMLA_HD inline int find_request(const SchedParams& sp, int64_t P, int VB, int64_t x) {
  int lo = 0, hi = VB - 1;
  if (sched_mode<MODE>(sp) == kSchedCascade) {
    const int VP = sched_prefix_units(sp);
    const int64_t unit_p = static_cast<int64_t>(sp.groups) *
                           (sched_piece_cost(sp) + sched_weight<MODE>(sp, 0) * P);
    if (x < unit_p * VP) return static_cast<int>(x / unit_p);
    lo = VP;
  }
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(sp.groups) * sched_line<MODE>(sp, P, mid) <= x)
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
template <int MODE = kSchedAny>
struct PieceIterT {
  SchedParams sp;
  int cta;
  int VB;
  int64_t P;
  int64_t W;
  int Gp;
  int64_t x, x1;       // auto policy cursor (cost-line points)
  int64_t p, p_end;    // fixed policy cursor
  Piece held;          // returned again by the next call of next() when have_held
  bool have_held;

  // Every member is assigned on every path: the iterator is only ever constructed with
  // init(), never copied.
  PMLA_HD void init(const SchedParams& s, int cta_id) {
    sp = s;
    cta = cta_id;
    P = sched_shared<MODE>(s);
    VB = sched_requests<MODE>(s);
    W = 0;
    Gp = 0;
    x = x1 = 0;
    p = p_end = 0;
    have_held = false;
    held = Piece{0, 0, 0, 0, 0, 0, 0, 0, 0, false, 0, 0};
    if (sp.splits <= 0) {
      W = static_cast<int64_t>(sp.groups) * (VB > 0 ? sched_line<MODE>(sp, P, VB) : 0);
      Gp = auto_ctas(static_cast<int64_t>(sp.groups) * (VB > 0 ? sched_cum<MODE>(sp, P, VB) : 0),
                     sp.grid);
      if (W <= 0 || cta >= Gp) {
        x = x1 = 0;
      } else {
        x = W * cta / Gp;
        x1 = W * (cta + 1) / Gp;
      }
    } else {
      p = cta;
      p_end = static_cast<int64_t>(VB) * sp.groups * sp.splits;
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
        const int v = find_request<MODE>(sp, P, VB, x);
        const int64_t base = static_cast<int64_t>(sp.groups) * sched_line<MODE>(sp, P, v);
        const int L = sched_len<MODE>(sp, P, v);
        const int64_t e = sched_piece_cost(sp);
        const int64_t w = sched_weight<MODE>(sp, v);
        const int64_t seg = e + w * (L > 0 ? L : 0);   // one row group's segment
        const int64_t off = x - base;
        if (L < 0 || off < 0 || off >= seg * sp.groups) {
          *bad = 1;
          x = x1;
          return false;
        }
        if (L == 0) {   // an empty request: nothing to attend, skip its segments
          x = (base + seg * sp.groups < x1) ? base + seg * sp.groups : x1;
          continue;
        }
        const int g = static_cast<int>(off / seg);
        const int64_t s0 = base + static_cast<int64_t>(g) * seg;
        const int64_t xe = (s0 + seg < x1) ? s0 + seg : x1;
        const int j0 = line_positions(x - s0, e, w, L);
        const int Lr = sched_real_len<MODE>(sp, P, v);   // <= L: a paged cache's last page
        const int j1v = line_positions(xe - s0, e, w, L);
        const int j1 = j1v < Lr ? j1v : Lr;
        x = xe;
        pc.b = v;
        pc.g = g;
        pc.j0 = j0;
        pc.j1 = j1;
        pc.L = Lr;
        pc.slot = static_cast<int64_t>(cta) + static_cast<int64_t>(v) * sp.groups + g;
        pc.direct = (j0 == 0 && j1 == Lr);
      } else {
        if (p >= p_end) return false;
        const int64_t u = p / sp.splits;
        const int k = static_cast<int>(p - u * sp.splits);
        const int v = static_cast<int>(u / sp.groups);
        const int g = static_cast<int>(u - static_cast<int64_t>(v) * sp.groups);
        const int L = sched_real_len<MODE>(sp, P, v);
        if (L < 0) {
          *bad = 1;
          p = p_end;
          return false;
        }
        pc.b = v;
        pc.g = g;
        piece_bounds(L, sp.splits, k, &pc.j0, &pc.j1);
        pc.L = L;
        pc.slot = p;
        pc.direct = (sp.splits == 1);
        p += sp.grid;
      }
      // a cascade half never holds the whole answer of a request (P > 0)
      if (sched_mode<MODE>(sp) != kSchedWhole && P > 0) pc.direct = false;
      pc.kv0 = sched_kv0<MODE>(sp, P, pc.b);
      int qo1 = 0;
      sched_tokens<MODE>(sp, pc.b, &pc.qo0, &qo1);
      pc.T = qo1 - pc.qo0;
      pc.cfrom = sched_cfrom<MODE>(sp, pc.b, pc.L, pc.T);
      const int rows_req = pc.T * sp.H;
      int rows = rows_req - pc.g * sp.NG;
      if (rows > sp.NG) rows = sp.NG;
      pc.rows = rows;
      if (rows > 0 && pc.j1 > pc.j0) return true;
    }
  }
};
// Runtime-mode iterator (host simulation).
using PieceIter = PieceIterT<kSchedAny>;

// Number of partial slots a call needs for (virtual) requests VB (host and device agree
// on this bound).
PMLA_HD inline int64_t partial_slots(int VB, int groups, int splits, int grid) {
  const int64_t units = static_cast<int64_t>(VB) * groups;
  if (splits <= 0) return units + grid;
  if (splits == 1) return 0;
  return units * splits;
}

// Partials of unit (v, g) as the decode kernel wrote them: slots first .. first+count-1
// (fixed policy: some may be empty pieces, see piece_bounds).  Returns false when the
// unit needs no merge: it ran whole on one CTA (written directly) or has no positions.
// In the cascade modes (with a shared prefix) every unit's pieces are partials.
template <int MODE = kSchedAny>
PMLA_HD inline bool unit_partials(const SchedParams& sp, int v, int g, int64_t* first,
                                  int* count) {
  const int64_t P = sched_shared<MODE>(sp);
  const int mode = sched_mode<MODE>(sp);
  const int VB = sched_requests<MODE>(sp);
  const int L = sched_len<MODE>(sp, P, v);        // page-rounded: the line's geometry
  const int Lr = sched_real_len<MODE>(sp, P, v);  // positions the unit holds
  if (Lr <= 0) return false;
  const bool all_partial = mode != kSchedWhole && P > 0;
  const int64_t u = static_cast<int64_t>(v) * sp.groups + g;
  if (sp.splits <= 0) {
    // position j of (v, g) is line point s0 + e + w j; its piece is on the CTA owning it
    const int64_t W = static_cast<int64_t>(sp.groups) * sched_line<MODE>(sp, P, VB);
    const int Gp = auto_ctas(static_cast<int64_t>(sp.groups) * sched_cum<MODE>(sp, P, VB),
                             sp.grid);
    const int64_t e = sched_piece_cost(sp);
    const int64_t w = sched_weight<MODE>(sp, v);
    const int64_t s0 = static_cast<int64_t>(sp.groups) * sched_line<MODE>(sp, P, v) +
                       static_cast<int64_t>(g) * (e + w * L);
    const int i0 = auto_cta_of(s0 + e, W, Gp);
    const int i1 = auto_cta_of(s0 + e + w * (Lr - 1), W, Gp);
    if (i0 == i1 && !all_partial) return false;
    *first = static_cast<int64_t>(i0) + u;   // CTA i writes unit u's piece to slot i + u
    *count = i1 - i0 + 1;
    return true;
  }
  if (sp.splits == 1 && !all_partial) return false;
  *first = u * sp.splits;
  *count = sp.splits;
  return true;
}

}  // namespace pmla
