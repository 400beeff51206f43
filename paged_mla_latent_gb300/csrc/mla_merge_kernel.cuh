// Softmax-weighted merge of normalised partial results (o_i, lse_i):
//   M = max_i lse_i,  w_i = exp(lse_i - M),  o = sum w_i o_i / sum w_i,
//   lse = M + ln sum w_i;  partials with lse = -inf weigh nothing.
// "Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache": each partial answer carries the
// normalisation information that lets shards (or split-KV pieces) merge exactly.
//
// One block handles one (output row, head) and a slice of the 512 value columns.  Its 256
// threads are P partial lanes x 256/P column quads (4 columns, one float4, per thread); a
// thread takes partials p, p+P, ... with several loads in flight, keeping a running max,
// weight sum and weighted sum.  P is picked per launch from the partials per row: many
// partials (batch 1, long history) want many lanes and few columns per block, so that the
// partials are read in one round; few partials want wide column slices.  Used twice:
// after the decode kernel, for the units the scheduler split, and by the public merge of
// context-parallel shards with an explicit reduce map.
#pragma once

#include <cuda_bf16.h>

#include "mla_sched.cuh"
#include "ptx.cuh"

namespace pmla {

constexpr int kMergeThreads = 256;
constexpr int kMergeBlocksPerSm = 3;   // launch bound: registers for 3 resident blocks
constexpr int kMergeWarps = kMergeThreads / 32;

// Merge launch shape for n_rows merged rows of ~per_row partials each.
//   lanes >= 2: one row per block, P = lanes partial lanes (a block covers 1024 / P
//               columns, 2 = a whole 512-column row) with U = unroll loads in flight;
//   lanes == 1: one row per warp (eight per block), each lane folding all of the row's
//               partials for its 16 columns.
// Every merge block pays a fixed latency (row lookup, the wait for the decode grid, one
// round of loads, the combine), so the shape aims at one wave of resident blocks: P is the
// smallest power of two giving each lane one round of U = 4 loads, halved while the grid
// exceeds a wave (U = 8 where a lane then has more than four loads); rows too many for one
// block each, with few partials, take a warp each.
struct MergeShape {
  int lanes, unroll;
};
inline int merge_lanes_for(int64_t per_row, int unroll) {
  int lanes = 2;
  while (lanes < 64 && lanes * unroll < per_row) lanes *= 2;
  return lanes;
}
inline MergeShape merge_shape_for(int64_t per_row, int64_t n_rows, int sms) {
  // n_rows: the merged rows that do work (padding rows of a row group return at once)
  const int64_t wave = static_cast<int64_t>(sms) * kMergeBlocksPerSm;
  if (n_rows > wave && per_row <= 16) return {1, 2};
  int lanes = merge_lanes_for(per_row, 4);
  while (lanes > 2 && n_rows * (lanes / 2) > wave) lanes /= 2;
  return {lanes, lanes * 4 >= per_row ? 4 : 8};
}
// Blocks along x for n_rows merged rows.
inline int64_t merge_blocks_x(const MergeShape& ms, int64_t n_rows) {
  return ms.lanes == 1 ? (n_rows + kMergeWarps - 1) / kMergeWarps : n_rows;
}


struct MergeOut {
  void* o;
  int o_fp32;
  int64_t o_off;      // element offset of this (row, head) in o
  float* lse;         // element for this (row, head), or null
};

// Running softmax-weighted state: max m, weight sum w, weighted sum a (4 columns).
struct MergeState {
  float m, w;
  float4 a;
};

__device__ __forceinline__ void merge_combine(MergeState& x, float m2, float w2, float4 a2) {
  if (m2 == -INFINITY) return;            // nothing in the other state
  const float M = fmaxf(x.m, m2);
  const float f1 = (x.m == -INFINITY) ? 0.f : __expf(x.m - M);
  const float f2 = __expf(m2 - M);
  x.w = x.w * f1 + w2 * f2;
  x.a.x = x.a.x * f1 + a2.x * f2;
  x.a.y = x.a.y * f1 + a2.y * f2;
  x.a.z = x.a.z * f1 + a2.z * f2;
  x.a.w = x.a.w * f1 + a2.w * f2;
  x.m = M;
}

// Merge `count` partials of one (row, head) for columns col0 .. col0 + 1024/P - 1.
// lse_of(k) and o_of(k) give partial k's log-sum-exp and the start of its 512 normalised
// values.  Lanes of one warp that share a column quad combine by shuffles, the eight warps
// through shared memory.
template <int P, int U, class OOf, class LseOf>
__device__ void merge_partials_block(int count, OOf o_of, LseOf lse_of, const MergeOut& out,
                                     int col0) {
  constexpr int Q = kMergeThreads / P;    // column quads per block
  constexpr int kCols = 4 * Q;
  // Rows of partial states left after the in-warp combine: one per warp when a warp holds
  // several partial lanes of the same columns (Q < 32), else one per partial lane.
  constexpr int R = Q < 32 ? kMergeWarps : P;
  static_assert(Q * P == kMergeThreads && kCols <= kDV, "bad merge shape");
  __shared__ float s_m[R][Q];
  __shared__ float s_w[R][Q];
  __shared__ float4 s_acc[R][Q];
  const int c = threadIdx.x % Q;
  const int p = threadIdx.x / Q;
  MergeState st{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int k0 = p; k0 < count; k0 += U * P) {
    float l[U];
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + u * P;
      l[u] = (k < count) ? lse_of(k) : -INFINITY;
      v[u] = (k < count) ? *reinterpret_cast<const float4*>(o_of(k) + col0 + 4 * c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) merge_combine(st, l[u], 1.f, v[u]);
  }
  const int lane = threadIdx.x & 31;
  if constexpr (Q < 32) {
    // lanes q, q + Q, q + 2Q, ... of a warp hold the same columns
#pragma unroll
    for (int off = Q; off < 32; off <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, st.m, off);
      const float w2 = __shfl_xor_sync(0xffffffffu, st.w, off);
      float4 a2;
      a2.x = __shfl_xor_sync(0xffffffffu, st.a.x, off);
      a2.y = __shfl_xor_sync(0xffffffffu, st.a.y, off);
      a2.z = __shfl_xor_sync(0xffffffffu, st.a.z, off);
      a2.w = __shfl_xor_sync(0xffffffffu, st.a.w, off);
      merge_combine(st, m2, w2, a2);
    }
    if (lane < Q) {
      const int w = threadIdx.x >> 5;
      s_m[w][lane] = st.m;
      s_w[w][lane] = st.w;
      s_acc[w][lane] = st.a;
    }
  } else {
    s_m[p][c] = st.m;
    s_w[p][c] = st.w;
    s_acc[p][c] = st.a;
  }
  __syncthreads();
  for (int col = threadIdx.x; col < kCols; col += kMergeThreads) {
    const int cq = col >> 2;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < R; ++w) M = fmaxf(M, s_m[w][cq]);
    float tot = 0.f, val = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < R; ++w) {
        if (s_m[w][cq] == -INFINITY) continue;
        const float f = __expf(s_m[w][cq] - M);
        tot += s_w[w][cq] * f;
        val += reinterpret_cast<const float*>(&s_acc[w][cq])[col & 3] * f;
      }
      val /= tot;
    }
    const int64_t off = out.o_off + col0 + col;
    if (out.o_fp32)
      reinterpret_cast<float*>(out.o)[off] = val;
    else
      reinterpret_cast<__nv_bfloat16*>(out.o)[off] = __float2bfloat16_rn(val);
    if (col == 0 && out.lse != nullptr && col0 == 0)
      *out.lse = (M == -INFINITY) ? -INFINITY : M + __logf(tot);
  }
}

// Merge `count` partials of one (row, head) with one warp: lane l owns columns
// 128 j + 4 l .. 128 j + 4 l + 3 (j = 0..3), so each load and store instruction of the warp
// covers 512 contiguous bytes of fp32 (256 of bf16).  All of a row's columns share one max
// and one weight sum, so the exponentials are taken once per partial.
template <int U, class OOf, class LseOf>
__device__ void merge_row_warp(int count, OOf o_of, LseOf lse_of, const MergeOut& out) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, w = 0.f;
  float4 a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < count; k0 += U) {
    float l[U];
    float4 v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + u;
      l[u] = (k < count) ? lse_of(k) : -INFINITY;
      const float* src = (k < count) ? o_of(k) : nullptr;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[u][j] = (k < count) ? *reinterpret_cast<const float4*>(src + 128 * j + 4 * lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (l[u] == -INFINITY) continue;
      const float M = fmaxf(m, l[u]);
      const float f1 = (m == -INFINITY) ? 0.f : __expf(m - M);
      const float f2 = __expf(l[u] - M);
      w = w * f1 + f2;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[j].x = a[j].x * f1 + v[u][j].x * f2;
        a[j].y = a[j].y * f1 + v[u][j].y * f2;
        a[j].z = a[j].z * f1 + v[u][j].z * f2;
        a[j].w = a[j].w * f1 + v[u][j].w * f2;
      }
      m = M;
    }
  }
  const float inv = (m == -INFINITY) ? 0.f : 1.f / w;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 r = make_float4(a[j].x * inv, a[j].y * inv, a[j].z * inv, a[j].w * inv);
    const int64_t off = out.o_off + 128 * j + 4 * lane;
    if (out.o_fp32) {
      float* d = reinterpret_cast<float*>(out.o) + off;
      if ((reinterpret_cast<uintptr_t>(d) & 15) == 0) {
        *reinterpret_cast<float4*>(d) = r;
      } else {
        d[0] = r.x; d[1] = r.y; d[2] = r.z; d[3] = r.w;
      }
    } else {
      __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(out.o) + off;
      const __nv_bfloat162 lo2 = __floats2bfloat162_rn(r.x, r.y);
      const __nv_bfloat162 hi2 = __floats2bfloat162_rn(r.z, r.w);
      if ((reinterpret_cast<uintptr_t>(d) & 7) == 0) {
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo2);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(d) = pk;
      } else {
        d[0] = lo2.x; d[1] = lo2.y; d[2] = hi2.x; d[3] = hi2.y;
      }
    }
  }
  if (lane == 0 && out.lse != nullptr) *out.lse = (m == -INFINITY) ? -INFINITY : m + __logf(w);
}

// Wait until the grid this one depends on (launched before it on the stream with
// programmatic serialization) has completed and its writes are visible.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

struct SplitMergeParams {
  SchedParams sp;
  const float* part_o;     // (slots, NG, 512)
  const float* part_lse;   // (slots, NG)
  int64_t n_slots;
  void* o;
  int o_fp32;
  int64_t o_stride_tok, o_stride_head;
  float* lse_out;
  int64_t n_q_rows;
  int64_t n_merge_rows;    // units * NG
  int* err;
};

// grid = (merge_blocks_x(units * NG), P / 2), block = 256.  Merges the units the scheduler split and writes
// o = 0, lse = -inf for requests with no cache positions.  Units that ran whole on one
// CTA were written by the decode kernel and are skipped here.
template <int P, int U>
__global__ void __launch_bounds__(kMergeThreads, kMergeBlocksPerSm) mla_split_merge_kernel(const SplitMergeParams prm) {
  const SchedParams& sp = prm.sp;
  const int NG = sp.NG;
  // P = 1: merged row = warp (eight per block); else merged row = block
  const int64_t mrow = P == 1 ? static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5)
                              : static_cast<int64_t>(blockIdx.x);
  const bool lead = P == 1 ? (threadIdx.x & 31) == 0 : (threadIdx.x == 0 && blockIdx.y == 0);
  if (mrow >= prm.n_merge_rows) return;
  const int64_t u = mrow / NG;
  const int n = static_cast<int>(mrow - u * NG);
  const int b = static_cast<int>(u / sp.groups);
  const int g = static_cast<int>(u - static_cast<int64_t>(b) * sp.groups);
  const int col0 = P == 1 ? 0 : blockIdx.y * (4 * kMergeThreads / P);
  const int T = sp.qo_indptr[b + 1] - sp.qo_indptr[b];
  const int rows = T * sp.H - g * NG;
  if (n >= rows || n >= NG) return;
  const int L = sched_req_len<kSchedWhole>(sp, b);
  const int64_t r = static_cast<int64_t>(sp.qo_indptr[b]) * sp.H + static_cast<int64_t>(g) * NG + n;
  if (r < 0 || r >= prm.n_q_rows) {
    if (lead) atomicOr(prm.err, kErrMergeRow);
    return;
  }
  MergeOut out;
  out.o = prm.o;
  out.o_fp32 = prm.o_fp32;
  out.o_off = (r / sp.H) * prm.o_stride_tok + (r % sp.H) * prm.o_stride_head;
  out.lse = prm.lse_out ? prm.lse_out + r : nullptr;

  int64_t first = 0;
  int count = 0;
  if (L > 0) {
    if (!unit_partials<kSchedWhole>(sp, b, g, &first, &count)) return;   // written directly by its CTA
    if (first < 0 || first + count > prm.n_slots) {
      if (lead) atomicOr(prm.err, kErrMergeSlot);
      return;
    }
  }
  grid_dependency_wait();   // partials come from the decode kernel
  // (L == 0: no partial exists; count = 0 writes o = 0, lse = -inf)
  const int splits = sp.splits;
  auto o_of = [&](int k) -> const float* { return prm.part_o + ((first + k) * NG + n) * kDV; };
  auto lse_of = [&](int k) -> float {
    if (splits > 0) {   // fixed policy: piece k of a short unit may be empty
      int j0, j1;
      piece_bounds(L, splits, k, &j0, &j1);
      if (j1 <= j0) return -INFINITY;
    }
    return prm.part_lse[(first + k) * NG + n];
  };
  if constexpr (P == 1)
    merge_row_warp<U>(count, o_of, lse_of, out);
  else
    merge_partials_block<P, U>(count, o_of, lse_of, out, col0);
}

// ---------------------------------------------------------------- shared-prefix cascade

struct CascadeMergeParams {
  SchedParams sp;          // the cascade schedule (sp.NG rows per slot, one group per unit)
  const float* part_o;     // (slots, sp.NG, 512)
  const float* part_lse;   // (slots, sp.NG)
  int64_t n_slots;
  int rows_per_req;        // grid.x = B * rows_per_req (= max_seqlen_q * H)
  void* o;
  int o_fp32;
  int64_t o_stride_tok, o_stride_head;
  float* lse_out;
  int64_t n_q_rows;
  int64_t n_merge_rows;    // B * rows_per_req
  int* err;
};

// grid = (merge_blocks_x(B * rows_per_req), P / 2), block = 256.  Row rr of request b merges the partials
// of its group's prefix unit (at row (qo_b - qo_group) H + rr of the group's rows) with
// those of its own unit (row rr).
// M: kSchedCascade (pages of one token, no page arithmetic compiled in; the merge's
// set-up is on the critical path after the decode grid, and a runtime choice of the two
// made the c16 call 2 us longer) or kSchedCascadePaged.
template <int P, int U, int M>
__global__ void __launch_bounds__(kMergeThreads, kMergeBlocksPerSm) mla_cascade_merge_kernel(const CascadeMergeParams prm) {
  const SchedParams& sp = prm.sp;
  const int NG = sp.NG;
  const int64_t mrow = P == 1 ? static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5)
                              : static_cast<int64_t>(blockIdx.x);
  const bool lead = P == 1 ? (threadIdx.x & 31) == 0 : (threadIdx.x == 0 && blockIdx.y == 0);
  if (mrow >= prm.n_merge_rows) return;
  const int b = static_cast<int>(mrow / prm.rows_per_req);
  const int rr = static_cast<int>(mrow - static_cast<int64_t>(b) * prm.rows_per_req);
  const int col0 = P == 1 ? 0 : blockIdx.y * (4 * kMergeThreads / P);
  const int qo0 = sp.qo_indptr[b];
  const int T = sp.qo_indptr[b + 1] - qo0;
  if (rr >= T * sp.H) return;
  const int64_t r = static_cast<int64_t>(qo0) * sp.H + rr;
  if (r < 0 || r >= prm.n_q_rows) {
    if (lead) atomicOr(prm.err, kErrMergeRow);
    return;
  }
  const int64_t shared = sched_shared<M>(sp);
  const int VP = sched_prefix_units(sp);
  const int v = b / sp.gsize;
  const int L = sched_req_len<M>(sp, b);
  int64_t pf = 0, sf = 0;
  int pc = 0, sc = 0;
  if (!unit_partials<M>(sp, v, 0, &pf, &pc)) pc = 0;
  if (!unit_partials<M>(sp, VP + b, 0, &sf, &sc)) sc = 0;
  if (L - shared < T - 1 && lead)
    atomicOr(prm.err, kErrBadInput);   // a query would not see the whole shared prefix
  const int np = (qo0 - sp.qo_indptr[v * sp.gsize]) * sp.H + rr;
  if (np >= NG || rr >= NG || (pc > 0 && (pf < 0 || pf + pc > prm.n_slots)) ||
      (sc > 0 && (sf < 0 || sf + sc > prm.n_slots))) {
    if (lead) atomicOr(prm.err, kErrMergeSlot);
    return;
  }
  grid_dependency_wait();   // partials come from the decode kernel
  MergeOut out;
  out.o = prm.o;
  out.o_fp32 = prm.o_fp32;
  out.o_off = (r / sp.H) * prm.o_stride_tok + (r % sp.H) * prm.o_stride_head;
  out.lse = prm.lse_out ? prm.lse_out + r : nullptr;
  auto o_of = [&](int k) -> const float* {
    return k < pc ? prm.part_o + ((pf + k) * NG + np) * kDV
                  : prm.part_o + ((sf + (k - pc)) * NG + rr) * kDV;
  };
  auto lse_of = [&](int k) -> float {
    return k < pc ? prm.part_lse[(pf + k) * NG + np] : prm.part_lse[(sf + (k - pc)) * NG + rr];
  };
  if constexpr (P == 1)
    merge_row_warp<U>(pc + sc, o_of, lse_of, out);
  else
    merge_partials_block<P, U>(pc + sc, o_of, lse_of, out, col0);
}

struct CsrMergeParams {
  const float* o_parts;     // (P, H, 512), last dim contiguous
  int64_t op_stride_p, op_stride_h;
  const float* lse_parts;   // (P, H)
  int64_t lp_stride_p, lp_stride_h;
  int64_t P;
  int H;
  const int32_t* reduce_indptr;
  const int32_t* reduce_idx;
  void* o;
  int o_fp32;
  int64_t o_stride_r, o_stride_h;
  float* lse_out;           // (n_out, H) contiguous or null
  int* err;
};

// grid = (n_out * H, P / 2), block = 256.  Public merge with an explicit reduce map.
template <int P>
__global__ void __launch_bounds__(kMergeThreads, kMergeBlocksPerSm) mla_csr_merge_kernel(const CsrMergeParams prm) {
  const int64_t rr = blockIdx.x / prm.H;
  const int h = static_cast<int>(blockIdx.x - rr * prm.H);
  const int col0 = blockIdx.y * (4 * kMergeThreads / P);
  const int beg = prm.reduce_indptr[rr];
  const int end = prm.reduce_indptr[rr + 1];
  const int count = end > beg ? end - beg : 0;
  MergeOut out;
  out.o = prm.o;
  out.o_fp32 = prm.o_fp32;
  out.o_off = rr * prm.o_stride_r + h * prm.o_stride_h;
  out.lse = prm.lse_out ? prm.lse_out + rr * prm.H + h : nullptr;
  auto slot = [&](int k) -> int64_t {
    const int64_t s = prm.reduce_idx[beg + k];
    return s;
  };
  auto o_of = [&](int k) -> const float* {
    int64_t s = slot(k);
    if (s < 0 || s >= prm.P) s = 0;   // flagged by lse_of, weight 0
    return prm.o_parts + s * prm.op_stride_p + h * prm.op_stride_h;
  };
  auto lse_of = [&](int k) -> float {
    const int64_t s = slot(k);
    if (s < 0 || s >= prm.P) {
      if (prm.err && (threadIdx.x & 31) == 0) atomicOr(prm.err, kErrMergeSlot);
      return -INFINITY;
    }
    return prm.lse_parts[s * prm.lp_stride_p + h * prm.lp_stride_h];
  };
  merge_partials_block<P, 4>(count, o_of, lse_of, out, col0);
}

struct ValidateParams {
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_lens;   // may be null (pages of one token)
  int log2_page;                   // kv_indptr counts pages of 2^log2_page tokens
  int B;
  int64_t n_q_tokens;
  int64_t kv_indices_len;
  int64_t n_kv_rows;
  int* err;
};

// Grid-stride check of the index inputs (debug path; never faults on bad data: every
// read is bounds-checked first).
__global__ void mla_validate_kernel(const ValidateParams prm) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int flags = 0;
  if (tid == 0) {
    if (prm.qo_indptr[0] != 0 || prm.qo_indptr[prm.B] != prm.n_q_tokens) flags |= kErrBadInput;
    if (prm.kv_indptr[0] < 0 || prm.kv_indptr[prm.B] > prm.kv_indices_len) flags |= kErrBadIndex;
  }
  for (int64_t b = tid; b < prm.B; b += nth) {
    const int T = prm.qo_indptr[b + 1] - prm.qo_indptr[b];
    const int pages = prm.kv_indptr[b + 1] - prm.kv_indptr[b];
    const int ps = 1 << prm.log2_page;
    const int last = prm.last_page_lens ? prm.last_page_lens[b] : 1;
    if (pages > 0 && (last < 1 || last > ps)) flags |= kErrBadInput;
    if (ps == 1 && last != 1) flags |= kErrBadInput;
    const int64_t L = pages > 0 ? (static_cast<int64_t>(pages) - 1) * ps + last : pages;
    if (T < 0 || L < 0 || L < T) flags |= kErrBadInput;
  }
  int64_t lo = prm.kv_indptr[0], hi = prm.kv_indptr[prm.B];
  if (lo < 0) lo = 0;
  if (hi > prm.kv_indices_len) hi = prm.kv_indices_len;
  for (int64_t j = lo + tid; j < hi; j += nth) {
    const int v = prm.kv_indices[j];
    if (v < 0 || v >= prm.n_kv_rows) flags |= kErrBadRowId;
  }
  if (flags) atomicOr(prm.err, flags);
}

}  // namespace pmla
