// The step after the decode: the 512-wide latent o of every (token, head) mapped to
// v_head_dim = 128 through that head's 512 x 128 matrix ("[Kimi-K3 MLA TP8] MLA
// performance", §2 geometry: kv_lora_rank 512, v_head_dim 128; §3: a separate batched
// matmul after the decode call).
//
//   v[t, h, n] = sum_{k<512} o[t, h, k] * w_uv[h, k, n]   (fp32 accumulation, bf16 result)
//
// A dense contraction, on the tensor cores with the operands swapped so that the matrix
// fills the MMA's M side: per head, v^T (128 x tokens) = w_uv[h]^T (128 x 512) . o^T
// (512 x tokens).  M = v_head_dim = 128 exactly, N = a tile of NT tokens (16 .. 256), so a
// decode batch of 16 tokens wastes nothing on M.  One CTA per (head, token tile):
//   warp 0   : TMA producer.  The K = 512 reduction runs in eight slices of 64: the matrix
//              slice (64 k rows x 128 n, MN-major, two 128-byte swizzled column chunks) and
//              the o slice (NT token rows x 64 k, K-major, 128-byte swizzle; rows past the
//              last token read zeros) land in eight stages (all in flight at once) for
//              tiles of up to 64 tokens, else in a ring of 6 (128 tokens) or 4 stages.
//   warp 1   : MMA issuer (tcgen05 kind::f16, bf16 x bf16, FP32 accumulator in TMEM: lane =
//              v column n, column = token), four K = 16 MMAs a slice.
//   warps 2-5: epilogue, TMEM lane quadrant (warp % 4): 16 tokens a load, bf16 stores.
// Every wait is bounded (2 s); a wait that runs out ends the CTA without writing v.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/paged_mla.h"
#include "mla_api_internal.h"
#include "ptx.cuh"

namespace pmla {
namespace {

constexpr int kVK = 512;                      // kv_lora_rank (the reduction)
constexpr int kVN = 128;                      // v_head_dim (the MMA's M)
constexpr int kKSlice = 64;                   // k per stage: one 128-byte row of bf16
constexpr int kSlices = kVK / kKSlice;        // 8
constexpr int kAChunkBytes = kKSlice * 128;   // 64 k rows x 64 n (128 B): 8 KB
constexpr int kASliceBytes = 2 * kAChunkBytes;
constexpr int kVThreads = 192;

template <int NT>
struct VLayout {
  static constexpr int kBSliceBytes = NT * 128;                  // NT token rows x 128 B
  static constexpr int kStageBytes = kASliceBytes + kBSliceBytes;  // multiple of 2 KB
  // up to 64 tokens every slice has its own stage (all eight loads in flight from the
  // start: one DRAM round trip); wider tiles cycle through a ring of 6 or 4
  static constexpr int kVStages = NT <= 64 ? kSlices : (NT == 128 ? 6 : 4);
  static constexpr int kBarOff = kVStages * kStageBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;             // + 1 KB alignment slack
  static constexpr int kTmemCols = NT < 32 ? 32 : NT;
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "MMA N");
  static_assert(kSmem <= 232448, "shared memory");
};

struct VProjParams {
  __nv_bfloat16* v;         // (n_tok, H, 128)
  int64_t v_st, v_sh;       // elements
  int64_t n_tok;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// D[tmem] (+)= A . B with bf16 operands and an FP32 accumulator, issued by one elected lane
// of a converged warp.
__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.b32 p, %4, 0, e;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16: D f32 ([4,6) = 1), A and B bf16 ([7,10) = [10,13) =
// 1), A MN-major ([15]), B K-major ([16] = 0), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// grid = (token tiles, H), block = 192.
template <int NT>
__global__ void __launch_bounds__(kVThreads, 1)
    mla_latent_to_v_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_o, const VProjParams p) {
  using LY = VLayout<NT>;
  constexpr int kVStages = LY::kVStages;
  extern __shared__ uint8_t smem_raw[];
  // the swizzled layouts need a 1024-byte aligned window
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  // barriers: full[S] (+0), empty[S] (+8 S), done (+16 S), drain (+16 S + 8); then the
  // TMEM base, the abort flag and a sink for the wait's error bit (no error word here)
  const uint32_t bars = sbase + LY::kBarOff;
  const uint32_t full0 = bars, empty0 = bars + 8 * kVStages, done = bars + 16 * kVStages;
  const uint32_t drain = done + 8;
  uint8_t* words = smem + LY::kBarOff + 16 * kVStages + 16;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(words);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(words + 4);
  int* err_sink = reinterpret_cast<int*>(words + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int t0 = blockIdx.x * NT;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_o);
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *err_sink = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), LY::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < kSlices; ++s) {
        const int st = s % kVStages;
        if (s >= kVStages &&
            !mbar_wait(empty0 + 8 * st, ((s / kVStages) - 1) & 1, abort_flag, err_sink))
          break;
        issued = s + 1;
        const uint32_t a = sbase + st * LY::kStageBytes;
        mbar_arrive_expect_tx(full0 + 8 * st, LY::kStageBytes);
        const int krow = h * kVK + s * kKSlice;
        tma_load_2d(a, &tm_w, 0, krow, full0 + 8 * st);                  // n 0 .. 63
        tma_load_2d(a + kAChunkBytes, &tm_w, 64, krow, full0 + 8 * st);  // n 64 .. 127
        tma_load_3d(a + kASliceBytes, &tm_o, s * kKSlice, h, t0, full0 + 8 * st);
      }
      // every load issued must land before the CTA may exit (they have, unless a wait ran
      // out): wait (bounded) for each stage's last fill
      for (int s = issued - kVStages > 0 ? issued - kVStages : 0; s < issued; ++s)
        mbar_wait_drain(full0 + 8 * (s % kVStages), (s / kVStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kVN, NT);
    bool ok = true;
    for (int s = 0; s < kSlices && ok; ++s) {
      const int st = s % kVStages;
      ok = warp_bcast(mbar_wait(full0 + 8 * st, (s / kVStages) & 1, abort_flag, err_sink));
      if (!ok) break;
      tc_fence_after();
      const uint32_t a = sbase + st * LY::kStageBytes;
      const uint32_t b = a + kASliceBytes;
#pragma unroll
      for (int j = 0; j < kKSlice / 16; ++j) {
        // A = w^T slice: M = 128 n in two 64-column chunks kAChunkBytes apart (leading
        // byte offset), 8-row k groups 1024 B apart (stride byte offset); 16 k rows per MMA.
        const uint64_t ad = smem_desc(a + j * 2048, kAChunkBytes, 1024, kSw128);
        // B = o^T slice: NT token rows of 128 B (K-major, 8-row groups 1024 B apart);
        // 16 k = 32 B per MMA inside the swizzled row.
        const uint64_t bd = smem_desc(b + j * 32, 16, 1024, kSw128);
        mma_bf16_warp(tmem, ad, bd, idesc, (s > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit_warp(empty0 + 8 * st);
    }
    if (ok) mma_commit_warp(done);
    // every MMA issued must finish before tensor memory is released (waited on below)
    mma_commit_warp(drain);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quadrant: n = 32 q + lane
    if (warp_bcast(mbar_wait(done, 0, abort_flag, err_sink))) {
      tc_fence_after();
      const int n = 32 * q + lane;
      __nv_bfloat16* vh = p.v + static_cast<int64_t>(h) * p.v_sh + n;
#pragma unroll 1
      for (int c = 0; c < NT / 16; ++c) {
        if (t0 + 16 * c >= p.n_tok) break;
        float x[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + 16 * c, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int64_t t = t0 + 16 * c + j;
          if (t < p.n_tok) vh[t * p.v_st] = __float2bfloat16_rn(x[j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait_drain(drain, 0);   // all issued MMAs complete (bounded)
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, LY::kTmemCols);
  }
}

template <int NT>
cudaError_t launch_vproj(const CUtensorMap& tw, const CUtensorMap& to, const VProjParams& p,
                         int H, cudaStream_t stream) {
  using LY = VLayout<NT>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(mla_latent_to_v_kernel<NT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  const dim3 grid(static_cast<unsigned>((p.n_tok + NT - 1) / NT), static_cast<unsigned>(H));
  mla_latent_to_v_kernel<NT><<<grid, kVThreads, LY::kSmem, stream>>>(tw, to, p);
  return cudaGetLastError();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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
  // o: the TMA view (512, H, n_tok) needs 16-byte strides and base
  if (o->stride[2] != 1 || o->stride[0] % 8 != 0 || o->stride[1] % 8 != 0 || o->stride[0] < 0 ||
      o->stride[1] < 0 || !aligned(o->ptr, 16))
    return MLA_ERR_INVALID_ARG;
  if (w_uv->stride[2] != 1 || w_uv->stride[1] != kVN || w_uv->stride[0] != kVK * kVN ||
      !aligned(w_uv->ptr, 16))
    return MLA_ERR_INVALID_ARG;
  if (v->stride[2] != 1 || v->stride[0] < 0 || v->stride[1] < 0 || !aligned(v->ptr, 2))
    return MLA_ERR_INVALID_ARG;
  if (n_tok >= (int64_t{1} << 31)) return MLA_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  // token tile: about one CTA per SM over (token tiles x heads), 16 .. 256 tokens, no wider
  // than the tokens there are
  int NT = 16;
  while (NT < 256 && static_cast<int64_t>(NT) * sms < n_tok * H) NT *= 2;
  while (NT > 16 && NT / 2 >= n_tok) NT /= 2;

  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!enc) return MLA_ERR_CUDA;
  CUtensorMap tw, to;
  {
    // the matrices as (H * 512 rows of k) x (128 n), box 64 n x 64 k, 128-byte swizzle
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kVN), static_cast<cuuint64_t>(H * kVK)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kVN * 2)};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kKSlice)};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uv->ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_INVALID_ARG;
  }
  {
    // o as (512 k, H, n_tok), box 64 k x 1 head x NT tokens; tokens past n_tok read zeros.
    // (A stride of a size-1 dimension is never stepped: any valid value will do.)
    const int64_t sh = H > 1 ? o->stride[1] : kVK;
    const int64_t st = n_tok > 1 ? o->stride[0] : H * sh;
    if (sh == 0 || st == 0) return MLA_ERR_INVALID_ARG;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kVK), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(n_tok)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(st * 2)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kKSlice), 1, static_cast<cuuint32_t>(NT)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o->ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_INVALID_ARG;
  }
  VProjParams p;
  p.v = static_cast<__nv_bfloat16*>(v->ptr);
  p.v_st = v->stride[0];
  p.v_sh = v->stride[1];
  p.n_tok = n_tok;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (NT) {
    case 16: e = launch_vproj<16>(tw, to, p, static_cast<int>(H), s); break;
    case 32: e = launch_vproj<32>(tw, to, p, static_cast<int>(H), s); break;
    case 64: e = launch_vproj<64>(tw, to, p, static_cast<int>(H), s); break;
    case 128: e = launch_vproj<128>(tw, to, p, static_cast<int>(H), s); break;
    default: e = launch_vproj<256>(tw, to, p, static_cast<int>(H), s); break;
  }
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
