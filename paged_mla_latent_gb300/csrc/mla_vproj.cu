// The step after the decode: the 512-wide latent o of every (token, head) mapped to
// v_head_dim = 128 through that head's 512 x 128 matrix ("[Kimi-K3 MLA TP8] MLA
// performance", §2 geometry: kv_lora_rank 512, v_head_dim 128; §3: a separate batched
// matmul after the decode call).
//
//   v[t, h, n] = sum_{k<512} o[t, h, k] * w_uv[h, k, n]   (fp32 accumulation, bf16 result)
//
// The work is small and bound by latency and L2: at 16 tokens x 12 heads it reads 1.5 MB
// of matrices and 192 KB of o.  One CTA takes one head and 16 output columns: it keeps
// that 512 x 16 slice of the head's matrix in shared memory and walks blocks of 16 tokens,
// each thread producing one (token, column) output with a 512-long dot product on the
// CUDA cores.  A tensor-core tile would waste most of its M side on 16 tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/paged_mla.h"

namespace pmla {
namespace {

constexpr int kVK = 512;       // kv_lora_rank
constexpr int kVN = 128;       // v_head_dim
constexpr int kVCols = 16;     // output columns per CTA
constexpr int kVTok = 16;      // tokens per block
constexpr int kVThreads = kVCols * kVTok;
constexpr int kVOPitch = kVK + 8;   // bf16 elements; 1,040 B rows put two token rows of a
                                    // warp on different banks
constexpr int kVMaxBlocksZ = 64;

struct VProjParams {
  const __nv_bfloat16* o;   // (n_tok, H, 512)
  int64_t o_st, o_sh;       // elements; multiples of 8
  const __nv_bfloat16* w;   // (H, 512, 128) contiguous
  __nv_bfloat16* v;         // (n_tok, H, 128)
  int64_t v_st, v_sh;       // elements
  int64_t n_tok;
  int H;
};

// grid = (128 / 16, H, token-block groups), block = 256.
__global__ void __launch_bounds__(kVThreads) mla_latent_to_v_kernel(const VProjParams p) {
  __shared__ __align__(16) __nv_bfloat16 ws[kVK][kVCols];    // 16 KB
  __shared__ __align__(16) __nv_bfloat16 os[kVTok][kVOPitch];  // 16.25 KB
  const int n0 = blockIdx.x * kVCols;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  // the head's 512 x 16 slice: two 16-byte pieces a row
  const __nv_bfloat16* wh = p.w + static_cast<int64_t>(h) * kVK * kVN + n0;
  for (int i = tid; i < kVK * 2; i += kVThreads) {
    const int k = i >> 1;
    const int half = i & 1;
    *reinterpret_cast<uint4*>(&ws[k][half * 8]) =
        __ldg(reinterpret_cast<const uint4*>(wh + static_cast<int64_t>(k) * kVN + half * 8));
  }
  const int tl = tid / kVCols;   // token within the block
  const int n = tid % kVCols;    // column within the slice
  for (int64_t t0 = static_cast<int64_t>(blockIdx.z) * kVTok; t0 < p.n_tok;
       t0 += static_cast<int64_t>(gridDim.z) * kVTok) {
    __syncthreads();   // the slice is in place / the previous block's reads are done
    for (int i = tid; i < kVTok * (kVK / 8); i += kVThreads) {
      const int tt = i / (kVK / 8);
      const int c = i % (kVK / 8);
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + tt < p.n_tok)
        val = __ldg(reinterpret_cast<const uint4*>(p.o + (t0 + tt) * p.o_st +
                                                   static_cast<int64_t>(h) * p.o_sh + c * 8));
      *reinterpret_cast<uint4*>(&os[tt][c * 8]) = val;
    }
    __syncthreads();
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
    for (int k = 0; k < kVK; k += 2) {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&os[tl][k]));
      acc0 = fmaf(of.x, __bfloat162float(ws[k][n]), acc0);
      acc1 = fmaf(of.y, __bfloat162float(ws[k + 1][n]), acc1);
    }
    if (t0 + tl < p.n_tok)
      p.v[(t0 + tl) * p.v_st + static_cast<int64_t>(h) * p.v_sh + n0 + n] =
          __float2bfloat16_rn(acc0 + acc1);
  }
}

bool aligned(const void* ptr, uintptr_t a) { return reinterpret_cast<uintptr_t>(ptr) % a == 0; }

}  // namespace
}  // namespace pmla

extern "C" int mla_latent_to_v(const mla_tensor_t* o, const mla_tensor_t* w_uv,
                               const mla_tensor_t* v, mla_stream_t stream) {
  using namespace pmla;
  if (!o || !w_uv || !v) return MLA_ERR_INVALID_ARG;
  if (o->ndim != 3 || w_uv->ndim != 3 || v->ndim != 3) return MLA_ERR_INVALID_ARG;
  if (o->dtype != MLA_DTYPE_BF16 || w_uv->dtype != MLA_DTYPE_BF16 || v->dtype != MLA_DTYPE_BF16)
    return MLA_ERR_INVALID_ARG;
  const int64_t n_tok = o->shape[0];
  const int64_t H = o->shape[1];
  if (n_tok < 0 || H < 1 || H > 65535) return MLA_ERR_INVALID_ARG;
  if (o->shape[2] != kVK || w_uv->shape[0] != H || w_uv->shape[1] != kVK ||
      w_uv->shape[2] != kVN || v->shape[0] != n_tok || v->shape[1] != H || v->shape[2] != kVN)
    return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  if (!o->ptr || !w_uv->ptr || !v->ptr) return MLA_ERR_INVALID_ARG;
  // o: 16-byte loads of 8 latent columns
  if (o->stride[2] != 1 || o->stride[0] % 8 != 0 || o->stride[1] % 8 != 0 || o->stride[0] < 0 ||
      o->stride[1] < 0 || !aligned(o->ptr, 16))
    return MLA_ERR_INVALID_ARG;
  if (w_uv->stride[2] != 1 || w_uv->stride[1] != kVN || w_uv->stride[0] != kVK * kVN ||
      !aligned(w_uv->ptr, 16))
    return MLA_ERR_INVALID_ARG;
  if (v->stride[2] != 1 || v->stride[0] < 0 || v->stride[1] < 0 || !aligned(v->ptr, 2))
    return MLA_ERR_INVALID_ARG;
  VProjParams p;
  p.o = static_cast<const __nv_bfloat16*>(o->ptr);
  p.o_st = o->stride[0];
  p.o_sh = o->stride[1];
  p.w = static_cast<const __nv_bfloat16*>(w_uv->ptr);
  p.v = static_cast<__nv_bfloat16*>(v->ptr);
  p.v_st = v->stride[0];
  p.v_sh = v->stride[1];
  p.n_tok = n_tok;
  p.H = static_cast<int>(H);
  const int64_t blocks = (n_tok + kVTok - 1) / kVTok;
  const dim3 grid(kVN / kVCols, static_cast<unsigned>(H),
                  static_cast<unsigned>(blocks < kVMaxBlocksZ ? blocks : kVMaxBlocksZ));
  mla_latent_to_v_kernel<<<grid, kVThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
