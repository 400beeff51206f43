// Softmax-weighted merge of normalised partial results (o_i, lse_i):
//   M = max_i lse_i,  w_i = exp(lse_i - M),  o = sum w_i o_i / sum w_i,
//   lse = M + ln sum w_i;  partials with lse = -inf weigh nothing.
// "Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache": each partial answer carries the
// normalisation information that lets shards (or split-KV pieces) merge exactly.
//
// One block handles one (output row, head) and a 128-column quarter of the 512 value
// columns.  Its 8 warps take the partials round-robin (lane = 4 columns, float4), each
// keeping a running max and weight sum; the warps are then combined through shared
// memory.  Used twice: after the decode kernel, for the units the scheduler split, and
// by the public merge of context-parallel shards with an explicit reduce map.
#pragma once

#include <cuda_bf16.h>

#include "mla_sched.cuh"
#include "ptx.cuh"

namespace pmla {

constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeCols = 32;           // value columns per block (one per lane)
constexpr int kMergeMaxParts = 1024;     // partials held in shared memory per pass

struct MergeOut {
  void* o;
  int o_fp32;
  int64_t o_off;      // element offset of this (row, head) in o
  float* lse;         // element for this (row, head), or null
};

// Merge `count` partials of one (row, head) for columns col0 .. col0+31.  lse_of(k) and
// o_of(k) give partial k's log-sum-exp and the start of its 512 normalised values.
// The block first turns the lse values into weights w_k = exp(lse_k - M) (shared by
// all its threads), then warp w accumulates partials w, w+8, ... with one column per lane,
// every load of a warp independent of the others.
template <class OOf, class LseOf>
__device__ void merge_partials_block(int count, OOf o_of, LseOf lse_of, const MergeOut& out,
                                     int col0) {
  __shared__ float s_w[kMergeMaxParts];
  __shared__ float s_red[kMergeWarps];
  __shared__ float s_acc[kMergeWarps][kMergeCols];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  float acc = 0.f, M = -INFINITY, wsum = 0.f;
  for (int base = 0; base < count || base == 0; base += kMergeMaxParts) {
    const int n = min(count - base, kMergeMaxParts);
    // 1. max of this pass's lse values
    float m = -INFINITY;
    for (int k = threadIdx.x; k < n; k += kMergeThreads) {
      const float l = lse_of(base + k);
      s_w[k] = l;
      m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float pm = s_red[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) pm = fmaxf(pm, s_red[w]);
    __syncthreads();
    if (pm == -INFINITY) continue;            // nothing attended in this pass
    // rescale what earlier passes accumulated to the new running max
    const float M_new = fmaxf(M, pm);
    const float f = (M == -INFINITY) ? 0.f : __expf(M - M_new);
    acc *= f;
    wsum *= f;
    M = M_new;
    // 2. weights
    for (int k = threadIdx.x; k < n; k += kMergeThreads) {
      const float l = s_w[k];
      s_w[k] = (l == -INFINITY) ? 0.f : __expf(l - M);
    }
    __syncthreads();
    float ws = 0.f;
    for (int k = lane; k < n; k += 32) ws += s_w[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    wsum += ws;   // every warp computes the same total
    // 3. weighted sum of the value rows: up to 8 independent loads in flight per warp
    float a = 0.f;
    for (int k0 = warp; k0 < n; k0 += 8 * kMergeWarps) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMergeWarps;
        v[u] = (k < n) ? o_of(base + k)[col0 + lane] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMergeWarps;
        if (k < n) a += s_w[k] * v[u];
      }
    }
    acc += a;
    __syncthreads();   // s_w is rewritten by the next pass
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (threadIdx.x < kMergeCols) {
    float val = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) val += s_acc[w][threadIdx.x];
    val = (wsum > 0.f) ? val / wsum : 0.f;
    const int64_t off = out.o_off + col0 + threadIdx.x;
    if (out.o_fp32)
      reinterpret_cast<float*>(out.o)[off] = val;
    else
      reinterpret_cast<__nv_bfloat16*>(out.o)[off] = __float2bfloat16_rn(val);
    if (threadIdx.x == 0 && out.lse != nullptr && col0 == 0)
      *out.lse = (wsum > 0.f) ? M + __logf(wsum) : -INFINITY;
  }
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
  int* err;
};

// grid = (units * NG, 512 / 32), block = 256.  Merges the units the scheduler split and writes
// o = 0, lse = -inf for requests with no cache positions.  Units that ran whole on one
// CTA were written by the decode kernel and are skipped here.
__global__ void __launch_bounds__(kMergeThreads) mla_split_merge_kernel(const SplitMergeParams prm) {
  const SchedParams& sp = prm.sp;
  const int NG = sp.NG;
  const int64_t u = blockIdx.x / NG;
  const int n = static_cast<int>(blockIdx.x - u * NG);
  const int b = static_cast<int>(u / sp.groups);
  const int g = static_cast<int>(u - static_cast<int64_t>(b) * sp.groups);
  const int col0 = blockIdx.y * kMergeCols;
  const int T = sp.qo_indptr[b + 1] - sp.qo_indptr[b];
  const int rows = T * sp.H - g * NG;
  if (n >= rows || n >= NG) return;
  const int L = sp.kv_indptr[b + 1] - sp.kv_indptr[b];
  const int64_t r = static_cast<int64_t>(sp.qo_indptr[b]) * sp.H + static_cast<int64_t>(g) * NG + n;
  if (r < 0 || r >= prm.n_q_rows) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(prm.err, kErrMergeRow);
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
    if (!unit_partials(sp, b, g, &first, &count)) return;   // written directly by its CTA
    if (first < 0 || first + count > prm.n_slots) {
      if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(prm.err, kErrMergeSlot);
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
  merge_partials_block(count, o_of, lse_of, out, col0);
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

// grid = (n_out * H, 512 / 32), block = 256.  Public merge with an explicit reduce map.
__global__ void __launch_bounds__(kMergeThreads) mla_csr_merge_kernel(const CsrMergeParams prm) {
  const int64_t rr = blockIdx.x / prm.H;
  const int h = static_cast<int>(blockIdx.x - rr * prm.H);
  const int col0 = blockIdx.y * kMergeCols;
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
  merge_partials_block(count, o_of, lse_of, out, col0);
}

struct ValidateParams {
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_lens;   // may be null
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
    const int L = prm.kv_indptr[b + 1] - prm.kv_indptr[b];
    if (T < 0 || L < 0 || L < T) flags |= kErrBadInput;
    if (prm.last_page_lens && prm.last_page_lens[b] != 1) flags |= kErrBadInput;
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
