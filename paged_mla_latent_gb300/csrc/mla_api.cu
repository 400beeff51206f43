// Host side of the C ABI declared in include/paged_mla.h: argument checks, workspace
// planning, TMA descriptors and kernel launches.  No device memory is allocated here;
// no host <-> device synchronisation happens except in mla_validate / mla_check_error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/paged_mla.h"
#include "mla_api_internal.h"
#include "mla_decode_launch.h"
#include "mla_merge_kernel.cuh"
#include "mla_sched.cuh"

namespace {

using namespace pmla;

constexpr size_t kHeaderBytes = 256;   // device error words live here
constexpr int kMaxDevices = 64;
constexpr int kMaxSeqlenQ = 64;
constexpr int kMaxHeads = 1024;
constexpr int kMaxPageSize = 1024;   // tokens per page (a power of two)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DeviceInfo {
  int sms = 0;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

int device_sms(int dev, int* sms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev[dev].sms == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
    g_dev[dev].sms = v;
  }
  *sms = g_dev[dev].sms;
  return MLA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D byte tensor (rows x 576) with the given row pitch; box = box_w x box_h.
int make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t pitch, int box_w, int box_h,
             CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_h)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 1-D contiguous int32 vector with at least `min_len` entries (or exactly `len` if len >= 0).
int check_i32_vec(const mla_tensor_t* t, int64_t len, int64_t* out_len) {
  if (!t || !t->ptr || t->dtype != MLA_DTYPE_INT32 || t->ndim != 1) return MLA_ERR_INVALID_ARG;
  if (t->shape[0] < 0 || (t->shape[0] > 1 && t->stride[0] != 1)) return MLA_ERR_INVALID_ARG;
  if (len >= 0 && t->shape[0] != len) return MLA_ERR_INVALID_ARG;
  if (!is_aligned(t->ptr, 4)) return MLA_ERR_INVALID_ARG;
  if (out_len) *out_len = t->shape[0];
  return MLA_OK;
}

int check_scalar_f32(const mla_tensor_t* t) {
  if (!t || !t->ptr || t->dtype != MLA_DTYPE_FP32) return MLA_ERR_INVALID_ARG;
  int64_t n = 1;
  for (int i = 0; i < t->ndim && i < 4; ++i) n *= t->shape[i];
  if (t->ndim < 0 || t->ndim > 4 || n != 1) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// Output o: (rows, H, 512) BF16/FP32, last dim contiguous.
int check_o(const mla_tensor_t* o, int64_t rows, int64_t H) {
  if (!o || !o->ptr || o->ndim != 3) return MLA_ERR_INVALID_ARG;
  if (o->dtype != MLA_DTYPE_BF16 && o->dtype != MLA_DTYPE_FP32) return MLA_ERR_INVALID_ARG;
  if (o->shape[0] != rows || o->shape[1] != H || o->shape[2] != kDV) return MLA_ERR_INVALID_ARG;
  if (o->stride[2] != 1 || o->stride[0] < 0 || o->stride[1] < 0) return MLA_ERR_INVALID_ARG;
  if (!is_aligned(o->ptr, o->dtype == MLA_DTYPE_FP32 ? 4 : 2)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int check_lse(const mla_tensor_t* l, int64_t rows, int64_t H) {
  if (!l) return MLA_OK;
  if (!l->ptr || l->dtype != MLA_DTYPE_FP32 || l->ndim != 2) return MLA_ERR_INVALID_ARG;
  if (l->shape[0] != rows || l->shape[1] != H) return MLA_ERR_INVALID_ARG;
  if ((H > 1 && l->stride[1] != 1) || (rows > 1 && l->stride[0] != H)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// Shared checks of q / kv_buffer / indptrs.  Fills the sizes it derives.
struct CallShape {
  int64_t n_tok = 0, H = 0, n_kv_rows = 0, kv_pitch = 0, kv_indices_len = 0;
  int64_t page_pitch = 0;   // bytes between pages (= kv_pitch for one-token pages)
  int log2_page = 0;        // pages of 2^log2_page tokens
  int B = 0;
};

int check_inputs(const mla_tensor_t* q, const mla_tensor_t* kv, const mla_tensor_t* qo_indptr,
                 const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                 const mla_tensor_t* last_page_lens, CallShape* cs) {
  if (!q || !q->ptr || q->dtype != MLA_DTYPE_FP8_E4M3FN || q->ndim != 3) return MLA_ERR_INVALID_ARG;
  if (q->shape[2] != kD) return MLA_ERR_UNSUPPORTED;
  if (q->shape[0] < 0 || q->shape[1] < 1 || q->shape[1] > kMaxHeads) return MLA_ERR_INVALID_ARG;
  if (q->stride[2] != 1 || q->stride[1] != kD || (q->shape[0] > 1 && q->stride[0] != q->shape[1] * kD))
    return MLA_ERR_INVALID_ARG;   // the TMA view of q needs it contiguous
  if (!is_aligned(q->ptr, 16)) return MLA_ERR_INVALID_ARG;
  cs->n_tok = q->shape[0];
  cs->H = q->shape[1];
  if (!kv || !kv->ptr || kv->dtype != MLA_DTYPE_FP8_E4M3FN) return MLA_ERR_INVALID_ARG;
  if (kv->ndim == 2) {
    if (kv->shape[1] != kD) return MLA_ERR_UNSUPPORTED;
    if (kv->stride[1] != 1) return MLA_ERR_INVALID_ARG;
    cs->kv_pitch = cs->page_pitch = kv->stride[0];
  } else if (kv->ndim == 4) {
    // (N_pages, page_size, nhead_kv = 1, 576): issue §4.1 kv_buffer shape, page_size 1 as
    // captured (§5.2) or a power of two up to kMaxPageSize (block-granular addressing)
    const int64_t ps = kv->shape[1];
    if (kv->shape[2] != 1 || kv->shape[3] != kD) return MLA_ERR_UNSUPPORTED;
    if (ps < 1 || ps > kMaxPageSize || (ps & (ps - 1)) != 0) return MLA_ERR_UNSUPPORTED;
    if (kv->stride[3] != 1) return MLA_ERR_INVALID_ARG;
    while ((int64_t{1} << cs->log2_page) < ps) ++cs->log2_page;
    cs->page_pitch = kv->stride[0];
    cs->kv_pitch = ps > 1 ? kv->stride[1] : kv->stride[0];
    if (ps > 1 && (cs->page_pitch % 16 != 0 || cs->page_pitch < (ps - 1) * cs->kv_pitch + kD))
      return MLA_ERR_INVALID_ARG;   // pages may not overlap
  } else {
    return MLA_ERR_INVALID_ARG;
  }
  cs->n_kv_rows = kv->shape[0];   // pages
  if (cs->n_kv_rows < 1 || (cs->n_kv_rows << cs->log2_page) >= 0x7FFFFFFF)
    return MLA_ERR_INVALID_ARG;   // virtual row ids (page * page_size + slot) fit int32
  if (cs->kv_pitch < kD || cs->kv_pitch % 16 != 0 || !is_aligned(kv->ptr, 16))
    return MLA_ERR_INVALID_ARG;   // 16-byte aligned base and row pitch
  int64_t nq = 0, nk = 0;
  int rc = check_i32_vec(qo_indptr, -1, &nq);
  if (rc) return rc;
  if (nq < 1) return MLA_ERR_INVALID_ARG;
  rc = check_i32_vec(kv_indptr, nq, &nk);
  if (rc) return rc;
  cs->B = static_cast<int>(nq - 1);
  rc = check_i32_vec(kv_indices, -1, &cs->kv_indices_len);
  if (rc) return rc;
  if (last_page_lens && last_page_lens->ptr) {
    rc = check_i32_vec(last_page_lens, cs->B, nullptr);
    if (rc) return rc;
  } else if (cs->log2_page > 0 && cs->B > 0) {
    return MLA_ERR_INVALID_ARG;   // with pages of several tokens the last page's fill is needed
  }
  return MLA_OK;
}

struct Plan {
  int NG, groups, grid, splits;
  int64_t slots;
  size_t lse_off, o_off, bytes;
  // Shared-prefix cascade (decode batches of <= 48 rows per request, at least one group):
  // cng-row tiles over gsize-request prefix units and per-request units, pslots partial
  // slots at plse_off / po_off (same header); cbytes = the larger of both layouts.
  bool cascade_ok;
  int cng;
  int gsize;
  int64_t pslots;
  size_t plse_off, po_off, cbytes;
};
// Rows of the cascade's tiles: 96 (the rows-on-lanes kernel) when a group of at least two
// requests fits and the batch fills one; else 48 for batches of 2..3 small requests.
constexpr int kPrefixNG = 96;
constexpr int kPrefixNGSmall = 48;

int make_plan(int B, int64_t H, int max_seqlen_q, int num_kv_splits, int sms, Plan* p) {
  if (B < 0 || H < 1 || H > kMaxHeads || max_seqlen_q < 1 || max_seqlen_q > kMaxSeqlenQ)
    return MLA_ERR_INVALID_ARG;
  if (sms < 1) return MLA_ERR_INVALID_ARG;
  const int rows = static_cast<int>(H * max_seqlen_q);
  p->NG = pick_group_rows(rows);
  p->groups = groups_for(rows, p->NG);
  p->grid = sms;
  p->splits = num_kv_splits <= 0 ? 0 : num_kv_splits;
  p->slots = partial_slots(B, p->groups, p->splits, p->grid);
  p->lse_off = kHeaderBytes;
  p->o_off = align_up(p->lse_off + static_cast<size_t>(p->slots) * p->NG * sizeof(float), 256);
  p->bytes = p->o_off + static_cast<size_t>(p->slots) * p->NG * kDV * sizeof(float);
  p->cascade_ok = false;
  p->cng = kPrefixNG;
  p->gsize = 1;
  p->pslots = 0;
  p->plse_off = p->po_off = p->bytes;
  p->cbytes = p->bytes;
  // (at least one full group: for fewer requests the extra launches cost more than
  // sharing the prefix saves)
  int cng = 0;
  if (rows <= kPrefixNG / 2 && B >= kPrefixNG / rows)
    cng = kPrefixNG;
  else if (rows <= kPrefixNGSmall / 2 && B >= kPrefixNGSmall / rows)
    cng = kPrefixNGSmall;
  if (p->splits == 0 && cng > 0) {
    p->cascade_ok = true;
    p->cng = cng;
    p->gsize = cng / rows;
    const int VP = (B + p->gsize - 1) / p->gsize;
    p->pslots = partial_slots(VP + B, 1, 0, p->grid);
    p->plse_off = kHeaderBytes;
    p->po_off = align_up(p->plse_off + static_cast<size_t>(p->pslots) * cng * sizeof(float), 256);
    const size_t end = p->po_off + static_cast<size_t>(p->pslots) * cng * kDV * sizeof(float);
    p->cbytes = end > p->bytes ? end : p->bytes;
  }
  return MLA_OK;
}

}  // namespace

namespace {

// Launch a merge kernel instantiation for (lanes, unroll) with programmatic dependent launch:
// the merge grid is scheduled while the decode grid runs and waits on the device
// (griddepcontrol.wait) for the partials.
template <int P, int U>
struct SplitMergeK {
  static void* fn() { return reinterpret_cast<void*>(mla_split_merge_kernel<P, U>); }
};
template <int P, int U>
struct CascadeMergeK {
  static void* fn() { return reinterpret_cast<void*>(mla_cascade_merge_kernel<P, U, kSchedCascade>); }
};
template <int P, int U>
struct CascadeMergePagedK {
  static void* fn() {
    return reinterpret_cast<void*>(mla_cascade_merge_kernel<P, U, kSchedCascadePaged>);
  }
};

template <template <int, int> class K>
void* merge_fn(const MergeShape& ms) {
  const bool u8 = ms.unroll == 8;
  switch (ms.lanes) {
    case 64: return u8 ? K<64, 8>::fn() : K<64, 4>::fn();
    case 32: return u8 ? K<32, 8>::fn() : K<32, 4>::fn();
    case 16: return u8 ? K<16, 8>::fn() : K<16, 4>::fn();
    case 8: return u8 ? K<8, 8>::fn() : K<8, 4>::fn();
    case 4: return u8 ? K<4, 8>::fn() : K<4, 4>::fn();
    case 2: return u8 ? K<2, 8>::fn() : K<2, 4>::fn();
    default: return K<1, 2>::fn();
  }
}

template <template <int, int> class K, class Params>
cudaError_t launch_merge(const MergeShape& ms, int64_t n_rows, const Params& mp, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(merge_blocks_x(ms, n_rows)), ms.lanes > 1 ? ms.lanes / 2 : 1);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<Params*>(&mp)};
  return cudaLaunchKernelExC(&cfg, merge_fn<K>(ms), args);
}

// Shared-prefix cascade: one launch of the plan.cng-row kernel over the prefix units (groups
// of plan.gsize requests attending the first `shared` positions) and the requests' own
// units, then the cascade merge of each row's two parts.
int launch_cascade(const Plan& plan, const DecodeParams& prm, const void* q_ptr, int64_t q_rows,
                   int32_t shared, int max_rows, cudaStream_t stream) {
  uint8_t* ws = reinterpret_cast<uint8_t*>(prm.err);
  int rc;
  CUtensorMap p_lat, p_rope;
  if ((rc = make_map(&p_lat, q_ptr, q_rows, kD, 128, plan.cng, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
  if ((rc = make_map(&p_rope, q_ptr, q_rows, kD, 64, plan.cng, CU_TENSOR_MAP_SWIZZLE_64B))) return rc;
  DecodeParams pp = prm;
  pp.sp.mode = pp.sp.log2_page > 0 ? kSchedCascadePaged : kSchedCascade;
  pp.sp.NG = plan.cng;
  pp.sp.groups = 1;
  pp.sp.gsize = plan.gsize;
  pp.sp.shared = shared;
  sched_set_costs(&pp.sp, max_rows);
  pp.part_lse = reinterpret_cast<float*>(ws + plan.plse_off);
  pp.part_o = reinterpret_cast<float*>(ws + plan.po_off);
  pp.n_slots = plan.pslots;
  rc = plan.cng == kPrefixNG ? launch_decode_ng96(p_lat, p_rope, pp, plan.grid, stream)
                             : launch_decode_ng48(p_lat, p_rope, pp, plan.grid, stream);
  if (rc) return rc;

  CascadeMergeParams mp;
  mp.sp = pp.sp;
  mp.part_o = pp.part_o;
  mp.part_lse = pp.part_lse;
  mp.n_slots = pp.n_slots;
  mp.rows_per_req = max_rows;
  mp.o = prm.o;
  mp.o_fp32 = prm.o_fp32;
  mp.o_stride_tok = prm.o_stride_tok;
  mp.o_stride_head = prm.o_stride_head;
  mp.lse_out = prm.lse_out;
  mp.n_q_rows = q_rows;
  mp.err = prm.err;
  const int B = prm.sp.B;
  mp.n_merge_rows = static_cast<int64_t>(B) * max_rows;
  const int VP = (B + plan.gsize - 1) / plan.gsize;
  const int64_t n_rows = static_cast<int64_t>(B) * max_rows;
  // partials per row: the CTAs one prefix unit spans plus those of the request's own unit
  // (the shape counts the rows that do work: q_rows <= n_rows)
  const MergeShape ms = merge_shape_for(plan.grid / VP + plan.grid / B + 4, q_rows, plan.grid);
  const cudaError_t e = pp.sp.mode == kSchedCascadePaged
                            ? launch_merge<CascadeMergePagedK>(ms, n_rows, mp, stream)
                            : launch_merge<CascadeMergeK>(ms, n_rows, mp, stream);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// mla_decode and mla_decode_shared_prefix: shared_len = the leading positions every
// request shares (0: none / unknown).  The cascade runs when the batch qualifies, the
// prefix is at least kMinShared long and the workspace holds the cascade's partials.
int decode_impl(const mla_tensor_t* q, const mla_tensor_t* kv_buffer, const mla_tensor_t* o,
                const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
                const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
                int32_t max_seqlen_q, float sm_scale, const mla_tensor_t* q_scale,
                const mla_tensor_t* kv_scale, int32_t num_kv_splits, int32_t shared_len,
                const mla_tensor_t* lse_out, void* workspace, size_t workspace_bytes,
                mla_stream_t stream_, bool check_only = false) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  CallShape cs;
  int rc = check_inputs(q, kv_buffer, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens, &cs);
  if (rc) return rc;
  if ((rc = check_o(o, cs.n_tok, cs.H))) return rc;
  if ((rc = check_lse(lse_out, cs.n_tok, cs.H))) return rc;
  if ((rc = check_scalar_f32(q_scale)) || (rc = check_scalar_f32(kv_scale))) return rc;
  if (!(sm_scale == sm_scale) || sm_scale == INFINITY || sm_scale == -INFINITY)
    return MLA_ERR_INVALID_ARG;
  if (max_seqlen_q < 1 || max_seqlen_q > kMaxSeqlenQ) return MLA_ERR_INVALID_ARG;
  if (shared_len < 0) return MLA_ERR_INVALID_ARG;
  if (!workspace || !is_aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  if (cs.B == 0 || cs.n_tok == 0) return MLA_OK;   // nothing to attend

  int dev = 0, sms = 0;
  if ((rc = current_device(&dev)) || (rc = device_sms(dev, &sms))) return rc;
  Plan plan;
  if ((rc = make_plan(cs.B, cs.H, max_seqlen_q, num_kv_splits, sms, &plan))) return rc;
  if (workspace_bytes < plan.bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (check_only) return MLA_OK;   // every host-side check passed; nothing enqueued

  CUtensorMap q_lat, q_rope;
  const int64_t q_rows = cs.n_tok * cs.H;
  if ((rc = make_map(&q_lat, q->ptr, q_rows, kD, 128, plan.NG, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
  if ((rc = make_map(&q_rope, q->ptr, q_rows, kD, 64, plan.NG, CU_TENSOR_MAP_SWIZZLE_64B))) return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams prm;
  prm.sp.kv_indptr = static_cast<const int32_t*>(kv_indptr->ptr);
  prm.sp.qo_indptr = static_cast<const int32_t*>(qo_indptr->ptr);
  prm.sp.B = cs.B;
  prm.sp.H = static_cast<int>(cs.H);
  prm.sp.NG = plan.NG;
  prm.sp.groups = plan.groups;
  prm.sp.splits = plan.splits;
  prm.sp.grid = plan.grid;
  prm.sp.mode = kSchedWhole;
  prm.sp.gsize = 1;
  prm.sp.shared = 0;
  sched_set_costs(&prm.sp, static_cast<int>(cs.H) * max_seqlen_q);
  prm.sp.log2_page = cs.log2_page;
  prm.sp.last_page_lens = (cs.log2_page > 0) ? static_cast<const int32_t*>(kv_last_page_lens->ptr)
                                             : nullptr;
  prm.kv = static_cast<const uint8_t*>(kv_buffer->ptr);
  prm.kv_pitch = cs.kv_pitch;
  prm.page_pitch = cs.page_pitch;
  prm.kv_indices = static_cast<const int32_t*>(kv_indices->ptr);
  prm.kv_indices_len = cs.kv_indices_len;
  prm.n_kv_rows = cs.n_kv_rows;
  prm.n_q_rows = q_rows;
  prm.q_scale = static_cast<const float*>(q_scale->ptr);
  prm.kv_scale = static_cast<const float*>(kv_scale->ptr);
  prm.sm_scale = sm_scale;
  prm.o = o->ptr;
  prm.o_fp32 = o->dtype == MLA_DTYPE_FP32;
  prm.o_stride_tok = o->stride[0];
  {
    // 16-byte stores cover 8 bf16 / 4 fp32 columns starting at a multiple of that count
    const int64_t run = o->dtype == MLA_DTYPE_FP32 ? 4 : 8;
    prm.o_vec16 = is_aligned(o->ptr, 16) && o->stride[0] % run == 0 && o->stride[1] % run == 0;
  }
  prm.o_stride_head = o->stride[1];
  prm.lse_out = lse_out ? static_cast<float*>(lse_out->ptr) : nullptr;
  prm.part_lse = reinterpret_cast<float*>(ws + plan.lse_off);
  prm.part_o = reinterpret_cast<float*>(ws + plan.o_off);
  prm.n_slots = plan.slots;
  prm.err = reinterpret_cast<int*>(ws);

  // On pages of several tokens the prefix units take the shared prefix's whole pages
  // (positions past the last whole page go with each request's own positions).
  const int32_t shared_whole = shared_len & ~((int32_t{1} << cs.log2_page) - 1);
  if (plan.cascade_ok && shared_whole >= kMinShared && workspace_bytes >= plan.cbytes)
    return launch_cascade(plan, prm, q->ptr, q_rows, shared_whole,
                          static_cast<int>(cs.H * max_seqlen_q), stream);

  switch (plan.NG) {
    case 16: rc = launch_decode_ng16(q_lat, q_rope, prm, plan.grid, stream); break;
    case 32: rc = launch_decode_ng32(q_lat, q_rope, prm, plan.grid, stream); break;
    case 48: rc = launch_decode_ng48(q_lat, q_rope, prm, plan.grid, stream); break;
    default: rc = launch_decode_ng96(q_lat, q_rope, prm, plan.grid, stream); break;
  }
  if (rc) return rc;

  SplitMergeParams mp;
  mp.sp = prm.sp;
  mp.part_o = prm.part_o;
  mp.part_lse = prm.part_lse;
  mp.n_slots = prm.n_slots;
  mp.o = prm.o;
  mp.o_fp32 = prm.o_fp32;
  mp.o_stride_tok = prm.o_stride_tok;
  mp.o_stride_head = prm.o_stride_head;
  mp.lse_out = prm.lse_out;
  mp.n_q_rows = q_rows;
  mp.err = prm.err;
  const int64_t units = static_cast<int64_t>(cs.B) * plan.groups;
  mp.n_merge_rows = units * plan.NG;
  // (rows past a group's real rows return at once: the shape counts the q_rows that work)
  const MergeShape ms = merge_shape_for(units > 0 ? plan.slots / units : 1, q_rows, plan.grid);
  const cudaError_t e = launch_merge<SplitMergeK>(ms, units * plan.NG, mp, stream);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

namespace pmla {

void* tensor_map_encoder() { return reinterpret_cast<void*>(encode_fn()); }

int check_decode_call(const mla_tensor_t* q, const mla_tensor_t* kv_buffer, const mla_tensor_t* o,
                      const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
                      const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
                      int32_t max_seqlen_q, float sm_scale, const mla_tensor_t* q_scale,
                      const mla_tensor_t* kv_scale, int32_t num_kv_splits,
                      const mla_tensor_t* lse_out, void* workspace, size_t workspace_bytes) {
  return decode_impl(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                     max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits, 0, lse_out,
                     workspace, workspace_bytes, nullptr, /*check_only=*/true);
}

}  // namespace pmla

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_BAD_INDEX: return "MLA_ERR_BAD_INDEX";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_BAD_INPUT: return "MLA_ERR_BAD_INPUT";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_get_workspace_size(int32_t batch_size, int32_t num_heads, int32_t max_seqlen_q,
                           int32_t num_kv_splits, int32_t num_sms, size_t* bytes_out) {
  if (!bytes_out) return MLA_ERR_INVALID_ARG;
  int sms = num_sms;
  if (sms <= 0) {
    int dev = 0;
    int rc = current_device(&dev);
    if (rc) return rc;
    rc = device_sms(dev, &sms);
    if (rc) return rc;
  }
  Plan p;
  int rc = make_plan(batch_size, num_heads, max_seqlen_q, num_kv_splits, sms, &p);
  if (rc) return rc;
  *bytes_out = p.bytes;
  return MLA_OK;
}

int mla_get_shared_prefix_workspace_size(int32_t batch_size, int32_t num_heads,
                                         int32_t max_seqlen_q, int32_t num_sms,
                                         size_t* bytes_out) {
  if (!bytes_out) return MLA_ERR_INVALID_ARG;
  int sms = num_sms;
  if (sms <= 0) {
    int dev = 0;
    int rc = current_device(&dev);
    if (rc) return rc;
    rc = device_sms(dev, &sms);
    if (rc) return rc;
  }
  Plan p;
  int rc = make_plan(batch_size, num_heads, max_seqlen_q, 0, sms, &p);
  if (rc) return rc;
  *bytes_out = p.cbytes;
  return MLA_OK;
}

int mla_decode(const mla_tensor_t* q, const mla_tensor_t* kv_buffer, const mla_tensor_t* o,
               const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
               const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
               int32_t max_seqlen_q, float sm_scale, const mla_tensor_t* q_scale,
               const mla_tensor_t* kv_scale, int32_t num_kv_splits, const mla_tensor_t* lse_out,
               void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  return decode_impl(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                     max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits, 0, lse_out,
                     workspace, workspace_bytes, stream);
}

int mla_decode_shared_prefix(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                             const mla_tensor_t* o, const mla_tensor_t* qo_indptr,
                             const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                             const mla_tensor_t* kv_last_page_lens, int32_t max_seqlen_q,
                             float sm_scale, const mla_tensor_t* q_scale,
                             const mla_tensor_t* kv_scale, int32_t shared_prefix_len,
                             const mla_tensor_t* lse_out, void* workspace,
                             size_t workspace_bytes, mla_stream_t stream) {
  return decode_impl(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                     max_seqlen_q, sm_scale, q_scale, kv_scale, 0, shared_prefix_len, lse_out,
                     workspace, workspace_bytes, stream);
}


int mla_merge_partials(const mla_tensor_t* o_parts, const mla_tensor_t* lse_parts,
                       const mla_tensor_t* reduce_indptr, const mla_tensor_t* reduce_idx,
                       const mla_tensor_t* o, const mla_tensor_t* lse_out, int32_t* error_word,
                       mla_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!o_parts || !o_parts->ptr || o_parts->dtype != MLA_DTYPE_FP32 || o_parts->ndim != 3)
    return MLA_ERR_INVALID_ARG;
  const int64_t P = o_parts->shape[0], H = o_parts->shape[1];
  if (o_parts->shape[2] != kDV || o_parts->stride[2] != 1 || H < 1 || H > kMaxHeads || P < 0)
    return MLA_ERR_INVALID_ARG;
  if (o_parts->stride[0] % 4 || o_parts->stride[1] % 4 || !is_aligned(o_parts->ptr, 16))
    return MLA_ERR_INVALID_ARG;   // rows are read as float4
  if (!lse_parts || !lse_parts->ptr || lse_parts->dtype != MLA_DTYPE_FP32 || lse_parts->ndim != 2 ||
      lse_parts->shape[0] != P || lse_parts->shape[1] != H)
    return MLA_ERR_INVALID_ARG;
  int64_t n1 = 0, m = 0;
  int rc = check_i32_vec(reduce_indptr, -1, &n1);
  if (rc) return rc;
  if (n1 < 1) return MLA_ERR_INVALID_ARG;
  if ((rc = check_i32_vec(reduce_idx, -1, &m))) return rc;
  const int64_t n_out = n1 - 1;
  if ((rc = check_o(o, n_out, H))) return rc;
  if ((rc = check_lse(lse_out, n_out, H))) return rc;
  if (n_out == 0) return MLA_OK;
  CsrMergeParams prm;
  prm.o_parts = static_cast<const float*>(o_parts->ptr);
  prm.op_stride_p = o_parts->stride[0];
  prm.op_stride_h = o_parts->stride[1];
  prm.lse_parts = static_cast<const float*>(lse_parts->ptr);
  prm.lp_stride_p = lse_parts->stride[0];
  prm.lp_stride_h = lse_parts->stride[1];
  prm.P = P;
  prm.H = static_cast<int>(H);
  prm.reduce_indptr = static_cast<const int32_t*>(reduce_indptr->ptr);
  prm.reduce_idx = static_cast<const int32_t*>(reduce_idx->ptr);
  prm.o = o->ptr;
  prm.o_fp32 = o->dtype == MLA_DTYPE_FP32;
  prm.o_stride_r = o->stride[0];
  prm.o_stride_h = o->stride[1];
  prm.lse_out = lse_out ? static_cast<float*>(lse_out->ptr) : nullptr;
  prm.err = error_word;
  const int lanes = merge_lanes_for(m / n_out, 4);
  dim3 grid(static_cast<unsigned>(n_out * H), lanes / 2);
  switch (lanes) {
    case 64: mla_csr_merge_kernel<64><<<grid, kMergeThreads, 0, stream>>>(prm); break;
    case 32: mla_csr_merge_kernel<32><<<grid, kMergeThreads, 0, stream>>>(prm); break;
    case 16: mla_csr_merge_kernel<16><<<grid, kMergeThreads, 0, stream>>>(prm); break;
    case 8: mla_csr_merge_kernel<8><<<grid, kMergeThreads, 0, stream>>>(prm); break;
    case 4: mla_csr_merge_kernel<4><<<grid, kMergeThreads, 0, stream>>>(prm); break;
    default: mla_csr_merge_kernel<2><<<grid, kMergeThreads, 0, stream>>>(prm); break;
  }
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_validate(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                 const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
                 const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
                 void* workspace, size_t workspace_bytes, mla_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  CallShape cs;
  int rc = check_inputs(q, kv_buffer, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens, &cs);
  if (rc) return rc;
  if (!workspace || workspace_bytes < kHeaderBytes || !is_aligned(workspace, 256))
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  int* word = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + sizeof(int));
  if (cudaMemsetAsync(word, 0, sizeof(int), stream) != cudaSuccess) return MLA_ERR_CUDA;
  ValidateParams prm;
  prm.qo_indptr = static_cast<const int32_t*>(qo_indptr->ptr);
  prm.kv_indptr = static_cast<const int32_t*>(kv_indptr->ptr);
  prm.kv_indices = static_cast<const int32_t*>(kv_indices->ptr);
  prm.last_page_lens = (kv_last_page_lens && kv_last_page_lens->ptr)
                           ? static_cast<const int32_t*>(kv_last_page_lens->ptr)
                           : nullptr;
  prm.log2_page = cs.log2_page;
  prm.B = cs.B;
  prm.n_q_tokens = cs.n_tok;
  prm.kv_indices_len = cs.kv_indices_len;
  prm.n_kv_rows = cs.n_kv_rows;
  prm.err = word;
  mla_validate_kernel<<<256, 256, 0, stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpyAsync(&host, word, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (host & (kErrBadIndex | kErrBadRowId)) return MLA_ERR_BAD_INDEX;
  if (host & kErrBadInput) return MLA_ERR_BAD_INPUT;
  return MLA_OK;
}

int mla_check_error(void* workspace, size_t workspace_bytes, mla_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!workspace || workspace_bytes < kHeaderBytes) return MLA_ERR_INVALID_ARG;
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (host == 0) return MLA_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (host & kErrTimeout) return MLA_ERR_TIMEOUT;
  if (host & kErrAnyIndex) return MLA_ERR_BAD_INDEX;
  if (host & kErrMisaligned) return MLA_ERR_UNSUPPORTED;
  if (host & kErrBadInput) return MLA_ERR_BAD_INPUT;
  return MLA_ERR_CUDA;
}

}  // extern "C"
