// mla_qk_rope_concat_and_cache: the step that produces the decode's inputs.
//
// "[Kimi-K3 MLA TP8] MLA performance" §3 "Entry point": the decode's q comes out of one
// fused step that rotates the rope part of q, places it after the 512 latent columns, and
// writes the step's new cache entry (512 latent + 64 rotated rope columns, §2 geometry)
// into the cache the decode then reads; q and the cache are float8_e4m3fn with per-tensor
// float32 scales (§4.1).  The rotary table is the caller's (row p = cos th_0..31, sin
// th_0..31 for position p) and the pairs are (2i, 2i+1) or (i, i+32).
//
// A memory-bound gather/scatter: one thread per 16 output bytes of one 576-byte output
// row (32 latent items, then 4 rope items), rows = every (token, head) of q plus one cache
// entry per token.  Loads and stores are 16 bytes, consecutive threads take consecutive
// 16-byte pieces of a row.  The arithmetic is the definition's, in fp32 with every
// operation rounded on its own (products, sum, quotient: no fused multiply-add), and the
// quotient goes to e4m3 in one rounding (cvt.rn.satfinite: nearest, ties to even,
// saturating at +-448), so the bytes are exact.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/paged_mla.h"
#include "ptx.cuh"

namespace {

constexpr int kItemsPerRow = 36;   // 32 latent pieces of 16 columns + 4 rope pieces
constexpr int kThreads = 256;

struct RopeCacheParams {
  const uint16_t* q_nope;   // bf16 bits
  int64_t qn_tok, qn_head;  // strides in elements
  const uint16_t* q_pe;
  int64_t qp_tok, qp_head;
  const uint16_t* kv_c;
  int64_t kc_tok;
  const uint16_t* k_pe;
  int64_t kp_tok;
  const int32_t* positions;
  const int32_t* slot_mapping;
  const float* cos_sin;
  int64_t cs_row;           // elements between table rows
  int64_t max_pos;
  int neox;
  const float* q_scale;
  const float* kv_scale;
  uint8_t* q_out;           // (n_tok, H, 576) contiguous
  uint8_t* kv;              // cache: slot s of page p at kv + p * page_pitch + s * slot_pitch
  int64_t page_pitch, slot_pitch;
  int log2_page;
  int64_t n_slots;          // N_pages << log2_page
  int64_t n_tok;
  int H;
  int* err;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Two fp32 values -> two e4m3fn codes (a in the low byte), nearest / ties to even,
// saturating at the largest finite value (NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// 16 bf16 values (two 16-byte words) divided by s, to 16 e4m3 codes (one 16-byte word).
__device__ __forceinline__ uint4 quantise16(const uint4& lo, const uint4& hi, float s) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
    const uint32_t c01 = e4m3x2(__fdiv_rn(bf16_bits_to_f32(w0 & 0xFFFFu), s),
                                __fdiv_rn(bf16_bits_to_f32(w0 >> 16), s));
    const uint32_t c23 = e4m3x2(__fdiv_rn(bf16_bits_to_f32(w1 & 0xFFFFu), s),
                                __fdiv_rn(bf16_bits_to_f32(w1 >> 16), s));
    out[i] = c01 | (c23 << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// The rotated pair (x c - y s, y c + x s), each product and the sum rounded to fp32.
__device__ __forceinline__ void rotate(float x, float y, float c, float s, float* ra, float* rb) {
  *ra = __fsub_rn(__fmul_rn(x, c), __fmul_rn(y, s));
  *rb = __fadd_rn(__fmul_rn(y, c), __fmul_rn(x, s));
}

__device__ __forceinline__ uint4 ld16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float4 ld16f(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// Rope piece r (0..3) of one row: a, b = its 16 bf16 rope values (interleaved pairs:
// columns 16r .. 16r+15; halves: x = columns 8r .. 8r+7, y = 32+8r .. 32+8r+7), cs = the
// token's table row, dst = the row's output columns 512.. .
__device__ __forceinline__ void rope_piece(const uint4& a, const uint4& b, const float* cs,
                                           int neox, int r, float scale, uint8_t* dst) {
  // cos and sin of the pair angles 8r .. 8r+7
  const float4 c0 = ld16f(cs + 8 * r), c1 = ld16f(cs + 8 * r + 4);
  const float4 s0 = ld16f(cs + 32 + 8 * r), s1 = ld16f(cs + 32 + 8 * r + 4);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  if (!neox) {
    // pairs (2i, 2i+1), i = 8r .. 8r+7: columns 16r .. 16r+15, one 16-byte output word
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float ra0, rb0, ra1, rb1;
      rotate(bf16_bits_to_f32(w[2 * k] & 0xFFFFu), bf16_bits_to_f32(w[2 * k] >> 16), c[2 * k],
             s[2 * k], &ra0, &rb0);
      rotate(bf16_bits_to_f32(w[2 * k + 1] & 0xFFFFu), bf16_bits_to_f32(w[2 * k + 1] >> 16),
             c[2 * k + 1], s[2 * k + 1], &ra1, &rb1);
      out[k] = e4m3x2(__fdiv_rn(ra0, scale), __fdiv_rn(rb0, scale)) |
               (e4m3x2(__fdiv_rn(ra1, scale), __fdiv_rn(rb1, scale)) << 16);
    }
    *reinterpret_cast<uint4*>(dst + 512 + 16 * r) = make_uint4(out[0], out[1], out[2], out[3]);
  } else {
    // pairs (i, i+32), i = 8r .. 8r+7: columns 8r .. 8r+7 and 32+8r .. 32+8r+7
    const uint32_t xw[4] = {a.x, a.y, a.z, a.w}, yw[4] = {b.x, b.y, b.z, b.w};
    uint32_t oa[2], ob[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = 2 * k + j;   // 16-bit pair of words: elements 2i, 2i+1
        rotate(bf16_bits_to_f32(xw[i] & 0xFFFFu), bf16_bits_to_f32(yw[i] & 0xFFFFu), c[2 * i],
               s[2 * i], &a[2 * j], &b[2 * j]);
        rotate(bf16_bits_to_f32(xw[i] >> 16), bf16_bits_to_f32(yw[i] >> 16), c[2 * i + 1],
               s[2 * i + 1], &a[2 * j + 1], &b[2 * j + 1]);
      }
      oa[k] = e4m3x2(__fdiv_rn(a[0], scale), __fdiv_rn(a[1], scale)) |
              (e4m3x2(__fdiv_rn(a[2], scale), __fdiv_rn(a[3], scale)) << 16);
      ob[k] = e4m3x2(__fdiv_rn(b[0], scale), __fdiv_rn(b[1], scale)) |
              (e4m3x2(__fdiv_rn(b[2], scale), __fdiv_rn(b[3], scale)) << 16);
    }
    *reinterpret_cast<uint2*>(dst + 512 + 8 * r) = make_uint2(oa[0], oa[1]);
    *reinterpret_cast<uint2*>(dst + 512 + 32 + 8 * r) = make_uint2(ob[0], ob[1]);
  }
}

__global__ void __launch_bounds__(kThreads) rope_cache_kernel(const RopeCacheParams p) {
  const int64_t items = p.n_tok * (p.H + 1) * kItemsPerRow;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t row = it / kItemsPerRow;
    const int k = static_cast<int>(it - row * kItemsPerRow);
    const int64_t t = row / (p.H + 1);
    const int h = static_cast<int>(row - t * (p.H + 1));
    const bool is_q = h < p.H;   // q row (t, h), else token t's new cache entry
    // Every load that depends on no other is issued before any result is used: the scale,
    // the position, the slot and the item's 32 source bytes (after an L2 flush each is a
    // DRAM round trip; in sequence they had tripled the kernel's time at 16 tokens).
    const float scale = __ldg(is_q ? p.q_scale : p.kv_scale);
    const int32_t pos = __ldg(p.positions + t);
    const int32_t slot = is_q ? 0 : __ldg(p.slot_mapping + t);
    const int r = k - 32;        // rope piece
    const uint16_t* src;
    int o1, o2;                  // element offsets of the two 16-byte source words
    if (k < 32) {
      src = is_q ? p.q_nope + t * p.qn_tok + h * p.qn_head : p.kv_c + t * p.kc_tok;
      o1 = 16 * k;
      o2 = 16 * k + 8;
    } else {
      src = is_q ? p.q_pe + t * p.qp_tok + h * p.qp_head : p.k_pe + t * p.kp_tok;
      o1 = p.neox ? 8 * r : 16 * r;
      o2 = p.neox ? 32 + 8 * r : 16 * r + 8;
    }
    const uint4 a = ld16(src + o1), b = ld16(src + o2);
    uint8_t* dst;
    if (is_q) {
      dst = p.q_out + (t * p.H + h) * 576;
    } else {
      if (slot < 0) continue;                   // no entry for this token
      if (static_cast<int64_t>(slot) >= p.n_slots) {
        if (k == 0) atomicOr(p.err, pmla::kErrBadRowId);
        continue;
      }
      const int64_t page = static_cast<int64_t>(slot) >> p.log2_page;
      const int64_t sl = slot & ((1 << p.log2_page) - 1);
      dst = p.kv + page * p.page_pitch + sl * p.slot_pitch;
    }
    if (k < 32) {
      *reinterpret_cast<uint4*>(dst + 16 * k) = quantise16(a, b, scale);
    } else {
      if (pos < 0 || static_cast<int64_t>(pos) >= p.max_pos) {
        if (h == 0 && k == 32) atomicOr(p.err, pmla::kErrBadIndex);
        continue;                               // rope columns left unwritten
      }
      rope_piece(a, b, p.cos_sin + static_cast<int64_t>(pos) * p.cs_row, p.neox, r, scale, dst);
    }
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// A bf16 tensor of `nd` dims with the given leading sizes and `inner` contiguous columns,
// 16-byte aligned, every other stride a non-negative multiple of 8 elements (16 bytes).
// (An empty tensor may have a null pointer.)
bool check_bf16(const mla_tensor_t* t, int nd, const int64_t* lead, int64_t inner) {
  if (!t || t->dtype != MLA_DTYPE_BF16 || t->ndim != nd) return false;
  if (!t->ptr && lead[0] != 0) return false;
  for (int i = 0; i + 1 < nd; ++i)
    if (t->shape[i] != lead[i] || t->stride[i] < 0 || t->stride[i] % 8 != 0) return false;
  return t->shape[nd - 1] == inner && t->stride[nd - 1] == 1 && aligned16(t->ptr);
}

bool check_i32(const mla_tensor_t* t, int64_t n) {
  return t && (t->ptr || n == 0) && t->dtype == MLA_DTYPE_INT32 && t->ndim == 1 && t->shape[0] == n &&
         (n <= 1 || t->stride[0] == 1) && (reinterpret_cast<uintptr_t>(t->ptr) & 3u) == 0;
}

bool check_scalar(const mla_tensor_t* t) {
  if (!t || !t->ptr || t->dtype != MLA_DTYPE_FP32 || t->ndim < 0 || t->ndim > 4) return false;
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n == 1;
}

}  // namespace

extern "C" int mla_qk_rope_concat_and_cache(
    const mla_tensor_t* q_nope, const mla_tensor_t* q_pe, const mla_tensor_t* kv_c,
    const mla_tensor_t* k_pe, const mla_tensor_t* positions, const mla_tensor_t* cos_sin,
    int32_t is_neox, const mla_tensor_t* slot_mapping, const mla_tensor_t* q_scale,
    const mla_tensor_t* kv_scale, const mla_tensor_t* q_out, const mla_tensor_t* kv_buffer,
    int32_t* error_word, mla_stream_t stream_) {
  if (!q_nope || q_nope->ndim != 3) return MLA_ERR_INVALID_ARG;
  const int64_t T = q_nope->shape[0], H = q_nope->shape[1];
  if (T < 0 || H < 1 || H > 1024) return MLA_ERR_INVALID_ARG;
  const int64_t th[2] = {T, H};
  if (!check_bf16(q_nope, 3, th, 512) || !check_bf16(q_pe, 3, th, 64)) return MLA_ERR_INVALID_ARG;
  if (!check_bf16(kv_c, 2, th, 512) || !check_bf16(k_pe, 2, th, 64)) return MLA_ERR_INVALID_ARG;
  if (!check_i32(positions, T) || !check_i32(slot_mapping, T)) return MLA_ERR_INVALID_ARG;
  if (!cos_sin || !cos_sin->ptr || cos_sin->dtype != MLA_DTYPE_FP32 || cos_sin->ndim != 2 ||
      cos_sin->shape[1] != 64 || cos_sin->shape[0] < 1 || cos_sin->stride[1] != 1 ||
      (cos_sin->shape[0] > 1 && (cos_sin->stride[0] < 64 || cos_sin->stride[0] % 4 != 0)) ||
      !aligned16(cos_sin->ptr))
    return MLA_ERR_INVALID_ARG;
  if (!check_scalar(q_scale) || !check_scalar(kv_scale)) return MLA_ERR_INVALID_ARG;
  if (is_neox != 0 && is_neox != 1) return MLA_ERR_INVALID_ARG;
  if (!q_out || (!q_out->ptr && T > 0) || q_out->dtype != MLA_DTYPE_FP8_E4M3FN || q_out->ndim != 3 ||
      q_out->shape[0] != T || q_out->shape[1] != H || q_out->shape[2] != 576 ||
      q_out->stride[2] != 1 || q_out->stride[1] != 576 || (T > 1 && q_out->stride[0] != H * 576) ||
      !aligned16(q_out->ptr))
    return MLA_ERR_INVALID_ARG;   // the decode's q layout: contiguous
  // the cache, as the decode takes it: (N, 576) or (N_pages, PS, 1, 576)
  const mla_tensor_t* kv = kv_buffer;
  if (!kv || !kv->ptr || kv->dtype != MLA_DTYPE_FP8_E4M3FN || !aligned16(kv->ptr))
    return MLA_ERR_INVALID_ARG;
  int64_t slot_pitch = 0, page_pitch = 0, ps = 1;
  if (kv->ndim == 2) {
    if (kv->shape[1] != 576 || kv->stride[1] != 1) return MLA_ERR_INVALID_ARG;
    slot_pitch = page_pitch = kv->stride[0];
  } else if (kv->ndim == 4) {
    ps = kv->shape[1];
    if (kv->shape[2] != 1 || kv->shape[3] != 576 || kv->stride[3] != 1) return MLA_ERR_INVALID_ARG;
    if (ps < 1 || ps > 1024 || (ps & (ps - 1)) != 0) return MLA_ERR_UNSUPPORTED;
    page_pitch = kv->stride[0];
    slot_pitch = ps > 1 ? kv->stride[1] : kv->stride[0];
    if (ps > 1 && page_pitch < (ps - 1) * slot_pitch + 576) return MLA_ERR_INVALID_ARG;
  } else {
    return MLA_ERR_INVALID_ARG;
  }
  if (kv->shape[0] < 1 || slot_pitch < 576 || slot_pitch % 16 != 0 || page_pitch % 16 != 0 ||
      (kv->shape[0] * ps) >= 0x7FFFFFFF)
    return MLA_ERR_INVALID_ARG;
  if (!error_word) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;

  RopeCacheParams p;
  p.q_nope = static_cast<const uint16_t*>(q_nope->ptr);
  p.qn_tok = q_nope->stride[0];
  p.qn_head = q_nope->stride[1];
  p.q_pe = static_cast<const uint16_t*>(q_pe->ptr);
  p.qp_tok = q_pe->stride[0];
  p.qp_head = q_pe->stride[1];
  p.kv_c = static_cast<const uint16_t*>(kv_c->ptr);
  p.kc_tok = kv_c->stride[0];
  p.k_pe = static_cast<const uint16_t*>(k_pe->ptr);
  p.kp_tok = k_pe->stride[0];
  p.positions = static_cast<const int32_t*>(positions->ptr);
  p.slot_mapping = static_cast<const int32_t*>(slot_mapping->ptr);
  p.cos_sin = static_cast<const float*>(cos_sin->ptr);
  p.cs_row = cos_sin->shape[0] > 1 ? cos_sin->stride[0] : 64;
  p.max_pos = cos_sin->shape[0];
  p.neox = is_neox;
  p.q_scale = static_cast<const float*>(q_scale->ptr);
  p.kv_scale = static_cast<const float*>(kv_scale->ptr);
  p.q_out = static_cast<uint8_t*>(q_out->ptr);
  p.kv = static_cast<uint8_t*>(kv->ptr);
  p.page_pitch = page_pitch;
  p.slot_pitch = slot_pitch;
  int lg = 0;
  while ((int64_t{1} << lg) < ps) ++lg;
  p.log2_page = lg;
  p.n_slots = kv->shape[0] * ps;
  p.n_tok = T;
  p.H = static_cast<int>(H);
  p.err = error_word;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  const int64_t items = T * (H + 1) * kItemsPerRow;
  int64_t blocks = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;   // 8 resident blocks of 256 a SM
  if (blocks > cap) blocks = cap;
  rope_cache_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                      reinterpret_cast<cudaStream_t>(stream_)>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
