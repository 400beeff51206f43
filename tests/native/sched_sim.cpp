// Host simulation of the split-KV schedule (test-suite only): runs the decode kernel's
// piece iterator for every CTA and the merge kernel's partial lookup for every unit,
// exactly as the device code does, and reports them to Python.
#include <stdint.h>

#include "../../paged_mla_latent_gb300/csrc/mla_sched.cuh"

extern "C" {

// Writes up to max_out pieces as 8 int64 each: cta, b, g, j0, j1, rows, slot, direct.
// Returns the number of pieces (or -1 if max_out was too small, -2 if an iterator
// reported inconsistent indptr data).
int64_t sched_pieces(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H, int NG,
                     int groups, int splits, int grid, int64_t* out, int64_t max_out) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid};
  int64_t n = 0;
  for (int cta = 0; cta < grid; ++cta) {
    pmla::PieceIter it;
    it.init(sp, cta);
    pmla::Piece pc;
    int bad = 0;
    while (it.next(pc, &bad)) {
      if (n >= max_out) return -1;
      int64_t* o = out + 8 * n;
      o[0] = cta; o[1] = pc.b; o[2] = pc.g; o[3] = pc.j0; o[4] = pc.j1; o[5] = pc.rows;
      o[6] = pc.slot; o[7] = pc.direct ? 1 : 0;
      ++n;
    }
    if (bad) return -2;
  }
  return n;
}

// For unit (b, g): returns 1 and first/count if it needs a merge, else 0.
int sched_unit_partials(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H, int NG,
                        int groups, int splits, int grid, int b, int g, int64_t* first,
                        int* count) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid};
  return pmla::unit_partials(sp, b, g, first, count) ? 1 : 0;
}

// Same for a cascade half: mode 1 = prefix (virtual requests of gsize requests), 2 =
// suffix; shared = the shared prefix length the device would have found.
int64_t sched_pieces_mode(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H, int NG,
                          int groups, int splits, int grid, int mode, int gsize, int shared,
                          int64_t* out, int64_t max_out) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared};
  int64_t n = 0;
  for (int cta = 0; cta < grid; ++cta) {
    pmla::PieceIter it;
    it.init(sp, cta);
    pmla::Piece pc;
    int bad = 0;
    while (it.next(pc, &bad)) {
      if (n >= max_out) return -1;
      int64_t* o = out + 10 * n;
      o[0] = cta; o[1] = pc.b; o[2] = pc.g; o[3] = pc.j0; o[4] = pc.j1; o[5] = pc.rows;
      o[6] = pc.slot; o[7] = pc.direct ? 1 : 0; o[8] = pc.kv0; o[9] = pc.cfrom;
      ++n;
    }
    if (bad) return -2;
  }
  return n;
}

int sched_unit_partials_mode(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                             int NG, int groups, int splits, int grid, int mode, int gsize,
                             int shared, int v, int g, int64_t* first, int* count) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared};
  return pmla::unit_partials(sp, v, g, first, count) ? 1 : 0;
}

// Any mode with explicit cost-line weights (w_own, w_prefix, piece_cost); 10 int64 per
// piece as sched_pieces_mode.
int64_t sched_pieces_cost(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H, int NG,
                          int groups, int splits, int grid, int mode, int gsize, int shared,
                          int w_own, int w_prefix, int piece_cost, int64_t* out, int64_t max_out) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared,
                       w_own, w_prefix, piece_cost};
  int64_t n = 0;
  for (int cta = 0; cta < grid; ++cta) {
    pmla::PieceIter it;
    it.init(sp, cta);
    pmla::Piece pc;
    int bad = 0;
    while (it.next(pc, &bad)) {
      if (n >= max_out) return -1;
      int64_t* o = out + 10 * n;
      o[0] = cta; o[1] = pc.b; o[2] = pc.g; o[3] = pc.j0; o[4] = pc.j1; o[5] = pc.rows;
      o[6] = pc.slot; o[7] = pc.direct ? 1 : 0; o[8] = pc.kv0; o[9] = pc.cfrom;
      ++n;
    }
    if (bad) return -2;
  }
  return n;
}

int sched_unit_partials_cost(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                             int NG, int groups, int splits, int grid, int mode, int gsize,
                             int shared, int w_own, int w_prefix, int piece_cost, int v, int g,
                             int64_t* first, int* count) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared,
                       w_own, w_prefix, piece_cost};
  return pmla::unit_partials(sp, v, g, first, count) ? 1 : 0;
}

// Paged caches: kv_indptr counts pages of 2^log2_page tokens, last_page_lens the last
// page's fill.  10 int64 per piece as sched_pieces_mode.
int64_t sched_pieces_paged(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                           int NG, int groups, int splits, int grid, int log2_page,
                           const int32_t* last_page_lens, int w_own, int piece_cost,
                           int64_t* out, int64_t max_out) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, 0, 1, 0,
                       w_own, 0, piece_cost, log2_page, last_page_lens};
  int64_t n = 0;
  for (int cta = 0; cta < grid; ++cta) {
    pmla::PieceIter it;
    it.init(sp, cta);
    pmla::Piece pc;
    int bad = 0;
    while (it.next(pc, &bad)) {
      if (n >= max_out) return -1;
      int64_t* o = out + 10 * n;
      o[0] = cta; o[1] = pc.b; o[2] = pc.g; o[3] = pc.j0; o[4] = pc.j1; o[5] = pc.rows;
      o[6] = pc.slot; o[7] = pc.direct ? 1 : 0; o[8] = pc.kv0; o[9] = pc.cfrom;
      ++n;
    }
    if (bad) return -2;
  }
  return n;
}

int sched_unit_partials_paged(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                              int NG, int groups, int splits, int grid, int log2_page,
                              const int32_t* last_page_lens, int w_own, int piece_cost, int v,
                              int g, int64_t* first, int* count) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, 0, 1, 0,
                       w_own, 0, piece_cost, log2_page, last_page_lens};
  return pmla::unit_partials(sp, v, g, first, count) ? 1 : 0;
}

// Every field: any mode on a paged cache.  10 int64 per piece as sched_pieces_mode.
int64_t sched_pieces_full(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                          int NG, int groups, int splits, int grid, int mode, int gsize,
                          int shared, int w_own, int w_prefix, int piece_cost, int log2_page,
                          const int32_t* last_page_lens, int64_t* out, int64_t max_out) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared,
                       w_own, w_prefix, piece_cost, log2_page, last_page_lens};
  int64_t n = 0;
  for (int cta = 0; cta < grid; ++cta) {
    pmla::PieceIter it;
    it.init(sp, cta);
    pmla::Piece pc;
    int bad = 0;
    while (it.next(pc, &bad)) {
      if (n >= max_out) return -1;
      int64_t* o = out + 10 * n;
      o[0] = cta; o[1] = pc.b; o[2] = pc.g; o[3] = pc.j0; o[4] = pc.j1; o[5] = pc.rows;
      o[6] = pc.slot; o[7] = pc.direct ? 1 : 0; o[8] = pc.kv0; o[9] = pc.cfrom;
      ++n;
    }
    if (bad) return -2;
  }
  return n;
}

int sched_unit_partials_full(const int32_t* kv_indptr, const int32_t* qo_indptr, int B, int H,
                             int NG, int groups, int splits, int grid, int mode, int gsize,
                             int shared, int w_own, int w_prefix, int piece_cost, int log2_page,
                             const int32_t* last_page_lens, int v, int g, int64_t* first,
                             int* count) {
  pmla::SchedParams sp{kv_indptr, qo_indptr, B, H, NG, groups, splits, grid, mode, gsize, shared,
                       w_own, w_prefix, piece_cost, log2_page, last_page_lens};
  return pmla::unit_partials(sp, v, g, first, count) ? 1 : 0;
}

// Tokens request b holds, as the merge kernels read it.
int sched_request_len(const int32_t* kv_indptr, int log2_page, const int32_t* last_page_lens,
                      int b) {
  pmla::SchedParams sp{};
  sp.kv_indptr = kv_indptr;
  sp.log2_page = log2_page;
  sp.last_page_lens = last_page_lens;
  return pmla::sched_req_len<pmla::kSchedAny>(sp, b);
}

// The weights the library sets for a call (mode, group rows NG, query rows per request).
void sched_host_costs(int mode, int NG, int rows_per_request, int* w_own, int* w_prefix,
                      int* piece_cost) {
  pmla::SchedParams sp{};
  sp.mode = mode;
  sp.NG = NG;
  pmla::sched_set_costs(&sp, rows_per_request);
  *w_own = sp.w_own;
  *w_prefix = sp.w_prefix;
  *piece_cost = sp.piece_cost;
}

int64_t sched_partial_slots(int B, int groups, int splits, int grid) {
  return pmla::partial_slots(B, groups, splits, grid);
}
}
