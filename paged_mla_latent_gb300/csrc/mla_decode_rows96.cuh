// Absorbed (latent) MLA decode with 96 query rows per pass over the cache, on sm_103a.
//
// What it computes is mla_decode_kernel's (mla_decode_kernel.cuh): "[Kimi-K3 MLA TP8] MLA
// performance" §2 (one 576-wide latent entry per token shared by every head, sm_scale =
// 1/sqrt(192)), §4.1 (fp8 q and cache, float32 q_scale / kv_scale), §5.2 (page-granular
// addressing); softmax partials and their merge: "Scaling Kimi K3 on AMD Instinct MI355X"
// §1 "Cache" and §4 "MLA".  This kernel serves groups of 49..96 query rows (a 96-head
// shard, or the shared prefix of eight 12-head requests) and reads every cache row once for
// all of them, where the 48-row kernel reads it once per 48 rows.
//
// Why a second design.  Tensor memory holds 128 lanes x 512 columns of 32 bits.  The other
// kernels keep positions on the lanes and O^T with the hi and lo planes of P side by side in
// N (2 x NG columns for each of four 128-wide value blocks), which caps NG at 48.  Here:
//   * QK puts the query rows on the lanes: S[n, j] = Q[n, :] . K[j, :] with q as the A
//     operand (M = 128 rows, 96 real) and the tile's cache rows as B (N = 64 positions),
//     both K-major, straight from the layouts the q load and the row gather write.
//   * PV stays O^T[c, n] += V^T[c, j] . P^T[j, n] (A = V^T read MN-major from the tile),
//     but the lo plane goes into the same accumulator as the hi plane: two block-scaled MMAs
//     (kind::mxf8f6f4) whose B scale factors are 1 and 2^-4.  O takes 4 x 96 columns.
//   * Tensor memory: O^T blocks at columns 0, 96, 192, 288; S (64 columns, one buffer) at
//     384; the constant scale factors at 448.
//   * A ring of four 64-position stages (shared memory: 4 x 36 KB of rows, 54 KB of q, two
//     P buffers of 12 KB).
//
// Warps: 0-2 and 5-7 gather rows as in mla_decode_kernel; warp 4 issues the QKs and warp 3
// the PVs (two issuers, so that one's waits overlap the other's MMAs); warps
// 8-15 are two softmax warpgroups: warp 8 + 4 h + q handles query rows 32 q .. 32 q + 31
// (TMEM lane quadrant q; q = 3 holds no rows) over positions 32 h .. 32 h + 31 of each tile,
// one row per thread, so a row's maximum and sum need no shuffles: the two halves exchange
// their tile maxima through shared memory at the tile's one barrier.  In the epilogue the
// eight warps read O^T (warp 8 + 4 h + q: value columns 32 q .. 32 q + 31 of blocks 2 h and
// 2 h + 1) and write o / lse or the normalised partials.
#pragma once

#include "mla_decode_kernel.cuh"

namespace pmla {

struct Rows96Layout {
  static constexpr int NG = 96;
  static constexpr int kTile = 64;                     // positions per tile
  static constexpr int STAGES = 4;
  static constexpr int kStageBytes = kTile * kD;       // 36,864
  static constexpr int kLatBlock = kTile * 128;        // one 128-column latent block of a stage
  static constexpr int kRopeOff = 4 * kLatBlock;       // rope block inside a stage
  static constexpr int kQOff = STAGES * kStageBytes;   // q tile: 4 latent blocks + rope block
  static constexpr int kQLatBlock = NG * 128;
  static constexpr int kQRopeOff = 4 * kQLatBlock;
  static constexpr int kQBytes = NG * kD;
  // P: two buffers (tile parity) of two planes (hi, lo), each kTile positions x NG rows,
  // K-major without swizzle: row n's bytes for positions 16 c .. 16 c + 15 at c * kPChunk
  // + 16 n.  (q's M = 128 QK reads 32 rows past each q block; past the rope block that is
  // the first 2 KB of P: don't-care rows of S.)
  static constexpr int kPChunk = NG * 16;
  static constexpr int kPPlane = kTile * NG;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kMiscOff = kPOff + 4 * kPPlane;
  // misc region (bytes from kMiscOff)
  static constexpr int kFull = 0;       // full[STAGES]
  static constexpr int kEmpty = 32;     // empty[STAGES]
  static constexpr int kSFull = 64;     // S written (one per tile)
  static constexpr int kSFree = 72;     // S read by every softmax warp (one per tile)
  static constexpr int kPFull = 80;     // p_full[2]
  static constexpr int kPv = 96;        // pv_done[2]
  static constexpr int kQFull = 112;
  static constexpr int kQEmpty = 120;
  static constexpr int kDrain = 128;     // QK issuer's MMAs done
  static constexpr int kTmemSlot = 136;
  static constexpr int kAbort = 140;
  static constexpr int kDrainPv = 144;   // PV issuer's MMAs done
  static constexpr int kRowOff = 192;                  // int64 output offset [NG]
  static constexpr int kXch = kRowOff + 8 * NG;        // float [tile parity][half][NG]
  static constexpr int kAlpha = kXch + 16 * NG;        // float rescale factor [NG]
  static constexpr int kScale = kAlpha + 4 * NG;       // float output scale [NG]
  static constexpr int kLPart = kScale + 4 * NG;       // float row sums [half][NG]
  static constexpr int kMiscBytes = kLPart + 8 * NG;
  static constexpr int kSmemBytes = kMiscOff + kMiscBytes;
  static_assert(kSmemBytes <= 232448, "shared memory overflow");
  static_assert(kStageBytes % 1024 == 0 && kLatBlock % 1024 == 0 && kQOff % 1024 == 0 &&
                    kQLatBlock % 1024 == 0 && kQRopeOff % 512 == 0,
                "swizzle atoms");
  static_assert(kQRopeOff + 128 * 64 <= kQBytes + 4 * kPPlane, "q over-read stays in shared memory");
  // tensor memory columns
  static constexpr int kOBase = 0;                     // O^T block b at kOBase + NG b
  static constexpr int kSCol = 4 * NG;                 // S: kTile columns
  static constexpr int kSfA = kSCol + kTile;           // scale factors of V (1)
  static constexpr int kSfHi = kSfA + 8;               // ... of P's hi plane (1)
  static constexpr int kSfLo = kSfA + 16;              // ... of P's lo plane (2^-4)
  static constexpr int kTmemCols = 512;
  static_assert(kSfLo + 8 <= kTmemCols, "tensor memory overflow");
  static constexpr int kThreads = 512;                 // 16 warps
  // Warps 0-2 and 5-7 gather rows, warp 4 issues QK, warp 3 issues PV.
  static constexpr int kProducers = 6;
  static constexpr int kQkWarp = 4;
  static constexpr int kPvWarp = 3;
  static constexpr int kRowsPerProducer = (kTile + kProducers - 1) / kProducers;   // 11
  // setmaxnreg: warpgroups 0-1 (producers, issuer) give registers to warpgroups 2-3
  static constexpr int kRegsLow = 96;
  static constexpr int kRegsHigh = 160;
  static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsHigh <= 65536, "register split");
};

// UE8M0 scale-factor bytes (2^(e - 127)), four to a tensor-memory column.
constexpr uint32_t kSf1x4 = 0x7F7F7F7Fu;       // 1
constexpr uint32_t kSfLo1x4 = 0x7B7B7B7Bu;     // 2^-4 = 1 / kLoScale
static_assert(kLoScale == 16.0f, "the lo plane's scale factor is 2^-4");

// Wait for a phase, polling with test_wait first: on a phase already complete that costs
// ~15 cycles against ~75 for try_wait (measured on GB300), and this kernel's issuing warp
// runs three such waits a tile between its MMAs.
__device__ __forceinline__ bool mbar_wait_test_first(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_flag, int* err) {
  if (mbar_test(bar, parity)) return true;
  return mbar_wait(bar, parity, abort_flag, err);
}

template <int MODE>
__global__ void __launch_bounds__(Rows96Layout::kThreads, 1)
    mla_decode_rows96_kernel(const __grid_constant__ CUtensorMap tm_q_lat,
                             const __grid_constant__ CUtensorMap tm_q_rope, const DecodeParams prm) {
  using LY = Rows96Layout;
  constexpr int NG = LY::NG;
  constexpr int STAGES = LY::STAGES;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t mbase = sbase + LY::kMiscOff;
  uint8_t* misc = smem + LY::kMiscOff;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc + LY::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + LY::kAbort);
  const uint32_t sQ = sbase + LY::kQOff;

  if ((sbase & 1023u) != 0) {   // the swizzled layouts need a 1024-byte aligned window
    if (threadIdx.x == 0) atomicOr(prm.err, kErrMisaligned);
    return;
  }
  if (threadIdx.x == 64) {
    prefetch_tensormap(&tm_q_lat);
    prefetch_tensormap(&tm_q_rope);
  }
  if (threadIdx.x < 64) {
    const int i = 32 * (threadIdx.x >> 1);
    if (i <= prm.sp.B) prefetch_l1((threadIdx.x & 1) ? prm.sp.qo_indptr + i : prm.sp.kv_indptr + i);
  }
  PieceIterT<MODE> iter;
  iter.init(prm.sp, blockIdx.x);
  int first_qrow;
  {
    Piece pc;
    int bad = 0;
    if (!iter.next(pc, &bad)) {    // no work for this CTA (uniform across the block)
      if (bad && threadIdx.x == 0) atomicOr(prm.err, kErrBadIndptr);
      return;
    }
    iter.hold(pc);
    first_qrow = pc.qo0 * prm.sp.H + pc.g * NG;
    if (threadIdx.x < LY::kTile / 32) {
      const int64_t gi = pc.kv0 + ((pc.j0 + 32 * threadIdx.x) >> prm.sp.log2_page);
      if (gi >= 0 && gi < prm.kv_indices_len) prefetch_l1(prm.kv_indices + gi);
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(mbase + LY::kFull + 8 * s, 32 * LY::kProducers);
      mbar_init(mbase + LY::kEmpty + 8 * s, 1);
    }
    mbar_init(mbase + LY::kSFull, 1);
    mbar_init(mbase + LY::kSFree, 8);          // every softmax warp
    for (int s = 0; s < 2; ++s) {
      mbar_init(mbase + LY::kPFull + 8 * s, 8);
      mbar_init(mbase + LY::kPv + 8 * s, 1);
    }
    mbar_init(mbase + LY::kQFull, 1);
    mbar_init(mbase + LY::kQEmpty, 1);
    mbar_init(mbase + LY::kDrain, 1);
    mbar_init(mbase + LY::kDrainPv, 1);
    *abort_flag = 0;
    fence_mbar_init();
    issue_q_load<NG>(sQ, &tm_q_lat, &tm_q_rope, first_qrow, mbase + LY::kQFull);
  }
  if (warp == LY::kQkWarp) {
    tmem_alloc(smem_u32(misc + LY::kTmemSlot), LY::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp >= kSoftmaxWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(LY::kRegsHigh));
    // ===================================================== softmax + epilogue (8 warps)
    const int hh = (warp - kSoftmaxWarp0) >> 2;   // tile positions 32 hh .. 32 hh + 31
    const int q4 = warp & 3;                      // TMEM lane quadrant
    const int n = 32 * q4 + lane;                 // query row of the group (q4 < 3) = S lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    if (hh == 0) {
      // the PV products' block-scale factors, constant for the kernel's life: 1 for V and
      // P's hi plane, 2^-4 for the lo plane (hi + lo / 16 in one accumulator)
      tmem_fill8(tl + LY::kSfA, kSf1x4);
      tmem_fill8(tl + LY::kSfHi, kSf1x4);
      tmem_fill8(tl + LY::kSfLo, kSfLo1x4);
      tmem_wait_st();
    }
    iter.init(prm.sp, blockIdx.x);
    const float kv_scale = *prm.kv_scale;
    const float scale_log2 = prm.sm_scale * (*prm.q_scale) * kv_scale * kLog2e;
    const int H = prm.sp.H;
    float* xch = reinterpret_cast<float*>(misc + LY::kXch);
    float* s_alpha = reinterpret_cast<float*>(misc + LY::kAlpha);
    float* s_scale = reinterpret_cast<float*>(misc + LY::kScale);
    float* l_part = reinterpret_cast<float*>(misc + LY::kLPart);
    int64_t* s_off = reinterpret_cast<int64_t*>(misc + LY::kRowOff);
    // this row's P vectors: positions 32 hh + 16 c' .. of buffer b, plane p at
    // kPOff + (2 b + p) kPPlane + (2 hh + c') kPChunk + 16 n
    uint8_t* prow = smem + LY::kPOff + 2 * hh * LY::kPChunk + 16 * n;
    constexpr int kBar = 1;   // named barrier of the 256 softmax threads

    uint32_t it_g = 0;
    Piece pc;
    while (iter.next(pc, &bad)) {
      const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
      const bool row_real = q4 < 3 && n < pc.rows;
      const bool warp_live = q4 < 3 && 32 * q4 < pc.rows;   // warp-uniform
      // Row n of the group is draft (g NG + n) / H of its request, which sees positions
      // <= cfrom + draft (prefix units: cfrom = L, no limit inside the piece).
      const int lim = pc.cfrom + (pc.g * NG + n) / H;
      const int vis_end = pc.j1 < lim + 1 ? pc.j1 : lim + 1;   // positions < vis_end are seen
      float m_ref = kRefInit;   // reference max - kPShift (log2 units)
      float l_acc = 0.f;        // this half's sum of p
      for (int t = 0; t < nt; ++t, ++it_g) {
        mbar_wait_test_first(mbase + LY::kSFull, it_g & 1, abort_flag, prm.err);
        tc_fence_after();
        float xs[32];
        if (warp_live) {
          tmem_ld32(tl + LY::kSCol + 32 * hh, xs);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(mbase + LY::kSFree);   // QK of the next tile may overwrite S
        // scaled logits (log2 units); positions past the piece, beyond the row's draft, or of
        // a padding row -> -inf
        float hmax = -INFINITY;
        if (warp_live) {
          const int pos0 = pc.j0 + t * LY::kTile + 32 * hh;
          int klim = row_real ? vis_end - pos0 : 0;
          klim = klim < 0 ? 0 : (klim > 32 ? 32 : klim);
          if (klim == 32) {
#pragma unroll
            for (int k = 0; k < 32; ++k) xs[k] *= scale_log2;
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) xs[k] = k < klim ? xs[k] * scale_log2 : -INFINITY;
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) hmax = fmaxf(hmax, xs[k]);
        }
        // the two halves' maxima meet at the tile's barrier; whether any row must move its
        // reference is decided there too (a half past the headroom <=> the row past it)
        float* xb = xch + (it_g & 1) * 2 * NG;
        if (q4 < 3) xb[hh * NG + n] = hmax;
        if (bar_red_or(kBar, 256, hmax - m_ref > kMoveAt)) {
          // rare: every row takes max(reference, tile max - kPShift)
          if (q4 < 3) {
            const float tmax = fmaxf(xb[n], xb[NG + n]);
            const float m_new = fmaxf(m_ref, tmax - kPShift);
            const float alpha = ex2_approx(m_ref - m_new);   // 0 from the initial reference
            l_acc *= alpha;
            m_ref = m_new;
            if (hh == 0) s_alpha[n] = alpha;
          }
          if (t > 0) {
            bar_sync(kBar, 256);   // every row's alpha is in shared memory
            // O holds this piece's earlier tiles: after the last PV, scale its row columns
            // (this warp: lanes 32 q4 .. of value blocks 2 hh, 2 hh + 1)
            mbar_wait(mbase + LY::kPv + 8 * ((it_g - 1) & 1), ((it_g - 1) >> 1) & 1, abort_flag,
                      prm.err);
            tc_fence_after();
#pragma unroll 1
            for (int bb = 0; bb < 2; ++bb) {
#pragma unroll 1
              for (int cg = 0; 32 * cg < pc.rows; ++cg) {
                float v[32];
                const uint32_t a = tl + LY::kOBase + (2 * hh + bb) * NG + 32 * cg;
                tmem_ld32(a, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] *= s_alpha[32 * cg + k];
                tmem_st32(a, v);
              }
            }
            tmem_wait_st();
          }
        }
        if (warp_live) {
          // scaled probabilities (<= 2^kMoveAt) as two FP8 planes: hi = e4m3(p),
          // lo = e4m3(kLoScale (p - hi)), the residual taken in f16x2
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float p0 = ex2_approx(xs[k] - m_ref);
            const float p1 = ex2_approx(xs[k + 1] - m_ref);
            l_acc += p0 + p1;
            const uint32_t p16 = f32x2_to_f16x2(p1, p0);   // low half: p0
            const uint32_t hi = f16x2_to_e4m3x2(p16);      // byte 0: p0, byte 1: p1
            const uint32_t r16 = f16x2_mul(f16x2_sub(p16, e4m3x2_to_f16x2(hi)), kLoScaleF16x2);
            const uint32_t lo = f16x2_to_e4m3x2(r16);
            if ((k & 2) == 0) {
              hw[k >> 2] = hi;
              lw[k >> 2] = lo;
            } else {
              hw[k >> 2] |= hi << 16;
              lw[k >> 2] |= lo << 16;
            }
          }
          // the buffer's previous tile (it_g - 2) must have been read by its PV: the PV
          // issuer is not ordered with the QK that signalled this tile's logits
          if (it_g >= 2)
            mbar_wait_test_first(mbase + LY::kPv + 8 * (it_g & 1), ((it_g - 2) >> 1) & 1,
                                 abort_flag, prm.err);
          uint8_t* pb = prow + (it_g & 1) * 2 * LY::kPPlane;
          *reinterpret_cast<uint4*>(pb) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(pb + LY::kPChunk) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          *reinterpret_cast<uint4*>(pb + LY::kPPlane) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          *reinterpret_cast<uint4*>(pb + LY::kPPlane + LY::kPChunk) =
              make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(mbase + LY::kPFull + 8 * (it_g & 1));
      }
      // ------------------------------------------------ piece epilogue
      {
        const uint32_t it_last = it_g - 1;
        if (q4 < 3) l_part[hh * NG + n] = l_acc;
        bar_sync(kBar, 256);
        const bool direct = pc.direct;
        const bool slot_ok = direct || (pc.slot >= 0 && pc.slot < prm.n_slots);
        if (hh == 0 && q4 < 3) {
          // one thread per row: normaliser, lse and output offset
          const float l = l_part[n] + l_part[NG + n];
          const float lse = (l > 0.f) ? (m_ref + lg2_approx(l)) * kLn2 : -INFINITY;
          int64_t off = -1;
          if (n < pc.rows) {
            if (direct) {
              const int rr = pc.g * NG + n;              // row within the request
              const int64_t tok = static_cast<int64_t>(pc.qo0) + rr / H;
              const int64_t r = tok * H + rr % H;
              if (r < prm.n_q_rows) {
                off = tok * prm.o_stride_tok + (rr % H) * prm.o_stride_head;
                if (prm.lse_out) prm.lse_out[r] = lse;
              } else {
                atomicOr(prm.err, kErrBadOutput);
              }
            } else if (slot_ok) {
              off = (pc.slot * NG + n) * kDV;
              prm.part_lse[pc.slot * NG + n] = lse;
            } else {
              atomicOr(prm.err, kErrBadOutput);
            }
          }
          s_scale[n] = (l > 0.f) ? kv_scale / l : 0.f;
          s_off[n] = off;
        }
        bar_sync(kBar, 256);
        mbar_wait(mbase + LY::kPv + 8 * (it_last & 1), (it_last >> 1) & 1, abort_flag, prm.err);
        tc_fence_after();
        // normalised output.  TMEM lane = value column: this warp holds value columns
        // 32 q4 .. 32 q4 + 31 of blocks 2 hh and 2 hh + 1 for every row; 16 rows at a time,
        // lanes exchange values (in-register transposes) so that each writes 16 contiguous
        // bytes of one row.  Scalar stores when o's layout does not allow 16-byte stores.
        const bool to_bf16 = direct && !prm.o_fp32;
        const bool vec = !direct || prm.o_vec16;
        float* fdst = direct ? reinterpret_cast<float*>(prm.o) : prm.part_o;
        __nv_bfloat16* hdst = reinterpret_cast<__nv_bfloat16*>(prm.o);
#pragma unroll 1
        for (int bb = 0; bb < 2; ++bb) {
          const int bk = 2 * hh + bb;
          const int cw = bk * 128 + 32 * q4;   // first value column of this warp
#pragma unroll 1
          for (int c0 = 0; c0 < pc.rows; c0 += 16) {
            float v[16];
            tmem_ld16(tl + LY::kOBase + bk * NG + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] *= s_scale[c0 + k];
            if (!vec) {
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const int64_t off = s_off[c0 + k];
                if (off < 0) continue;
                if (to_bf16)
                  hdst[off + cw + lane] = __float2bfloat16_rn(v[k]);
                else
                  fdst[off + cw + lane] = v[k];
              }
            } else if (to_bf16) {
              lane_transpose<8>(v, lane);
              lane_transpose<8>(v + 8, lane);
              const int cs = cw + 8 * (lane >> 3);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int64_t off = s_off[c0 + 8 * h + (lane & 7)];
                if (off >= 0) {
                  const float* a = v + 8 * h;
                  *reinterpret_cast<uint4*>(hdst + off + cs) =
                      make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                 pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
                }
              }
            } else {
#pragma unroll
              for (int g = 0; g < 4; ++g) lane_transpose<4>(v + 4 * g, lane);
              const int cs = cw + 4 * (lane >> 2);
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int64_t off = s_off[c0 + 4 * g + (lane & 3)];
                if (off >= 0)
                  *reinterpret_cast<float4*>(fdst + off + cs) =
                      make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
              }
            }
          }
        }
        bar_sync(kBar, 256);   // s_off / s_scale / l_part are rewritten by the next piece
        tc_fence_before();
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LY::kRegsLow));
    if (warp != LY::kQkWarp && warp != LY::kPvWarp) {
      // ===================================================== producers (6 warps)
      // As in mla_decode_kernel: producer pw copies tile rows r = pw + 6 j (j < rows_w), lane
      // j loads row j's id; 16-byte cp.async into the 128-byte (latent) / 64-byte (rope)
      // swizzled layouts.
      const int pw = warp < LY::kPvWarp ? warp : warp - 2;
      uint32_t it_g = 0;
      int n_piece = 0;
      int q_loads = 0;
      bool aborted = false;
      Piece pc;
      const uint8_t* kv = prm.kv;
      const int lg = prm.sp.log2_page;
      const int smask = (1 << lg) - 1;
      const int64_t ppitch = prm.page_pitch;
      const int64_t spitch = prm.kv_pitch;
      const int rows_w = (LY::kTile - pw + LY::kProducers - 1) / LY::kProducers;   // 11 / 10
      while (!aborted && iter.next(pc, &bad)) {
        const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
        if (warp == 0 && lane == 0) {
          if (n_piece == 0) {
            ++q_loads;
          } else if (!mbar_wait(mbase + LY::kQEmpty, (n_piece - 1) & 1, abort_flag, prm.err)) {
            aborted = true;
          } else {
            issue_q_load<NG>(sQ, &tm_q_lat, &tm_q_rope, pc.qo0 * prm.sp.H + pc.g * NG,
                             mbase + LY::kQFull);
            ++q_loads;
          }
        }
        aborted = __shfl_sync(0xffffffffu, aborted ? 1 : 0, 0) != 0;
        if (aborted) break;
        const int64_t kvbase = pc.kv0;
        auto load_row = [&](int t, int j) -> int64_t {
          if (j >= rows_w) return -1;
          const int pos = pc.j0 + t * LY::kTile + pw + LY::kProducers * j;
          if (pos >= pc.j1) return -1;
          const int64_t gi = kvbase + (pos >> lg);
          if (gi < 0 || gi >= prm.kv_indices_len) {
            atomicOr(prm.err, kErrBadIndex);
            return -1;
          }
          const int v = __ldg(prm.kv_indices + gi);
          if (v < 0 || static_cast<int64_t>(v) >= prm.n_kv_rows) {
            atomicOr(prm.err, kErrBadRowId);
            return -1;
          }
          return static_cast<int64_t>(v) * ppitch + static_cast<int64_t>(pos & smask) * spitch;
        };
        int64_t nxt = load_row(0, lane);
        for (int t = 0; t < nt; ++t, ++it_g) {
          const int stage = static_cast<int>(it_g % STAGES);
          const uint32_t use = it_g / STAGES;
          const uint32_t vmask = __ballot_sync(0xffffffffu, nxt >= 0);
          const int64_t rid = nxt >= 0 ? nxt : 0;
          if (t + 1 < nt) nxt = load_row(t + 1, lane);
          if (t + 2 < nt && lane < rows_w) {
            const int pos2 = pc.j0 + (t + 2) * LY::kTile + pw + LY::kProducers * lane;
            const int64_t gi = kvbase + (pos2 >> lg);
            if (gi >= 0 && gi < prm.kv_indices_len && pos2 < pc.j1) prefetch_l1(prm.kv_indices + gi);
          }
          constexpr bool kHoist = MODE == kSchedWhole;
          int64_t offs[kHoist ? LY::kRowsPerProducer : 1];
          if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < LY::kRowsPerProducer; ++j)
              offs[j] = __shfl_sync(0xffffffffu, rid, j);
          }
          if (use > 0 &&
              !mbar_wait(mbase + LY::kEmpty + 8 * stage, (use - 1) & 1, abort_flag, prm.err)) {
            aborted = true;
            break;
          }
          const uint32_t st = sbase + stage * LY::kStageBytes;
          const uint32_t blk = (lane >> 3) * LY::kLatBlock;
          const uint32_t chunk = lane & 7;
          if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < LY::kRowsPerProducer; ++j) {
              if (j < rows_w) {
                const int r = pw + LY::kProducers * j;
                const uint32_t dst = st + blk + r * 128 + ((chunk ^ (r & 7)) << 4);
                cp_async_16(dst, kv + offs[j] + 16 * lane, ((vmask >> j) & 1u) << 4);
              }
            }
          } else {
#pragma unroll 5
            for (int j = 0; j < rows_w; ++j) {
              const int r = pw + LY::kProducers * j;
              const int64_t off = __shfl_sync(0xffffffffu, rid, j);
              const uint32_t dst = st + blk + r * 128 + ((chunk ^ (r & 7)) << 4);
              cp_async_16(dst, kv + off + 16 * lane, ((vmask >> j) & 1u) << 4);
            }
          }
#pragma unroll
          for (int m = 0; m < (LY::kRowsPerProducer + 7) / 8; ++m) {
            const int j = 8 * m + (lane >> 2);
            const int c = lane & 3;
            const int64_t off = __shfl_sync(0xffffffffu, rid, j);
            if (j < rows_w) {
              const int r = pw + LY::kProducers * j;
              const uint32_t dst = st + LY::kRopeOff + r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
              cp_async_16(dst, kv + off + 512 + 16 * c, ((vmask >> j) & 1u) << 4);
            }
          }
          cp_async_arrive_noinc(mbase + LY::kFull + 8 * stage);
        }
        ++n_piece;
      }
      cp_async_wait_all();
      if (warp == 0 && lane == 0 && q_loads > 0)
        mbar_wait_drain(mbase + LY::kQFull, (q_loads - 1) & 1);
      __syncwarp();
    } else {
      // ===================================================== MMA issuers (two warps)
      // Warp 4 issues QK(0), QK(1), ... and warp 3 PV(0), PV(1), ... (CTA-wide tile
      // numbers), each waiting (bounded) only for its own inputs: QK(i) for its stage's rows,
      // the piece's q rows and S read by every softmax warp of tile i - 1 (one S buffer);
      // PV(i) for P(i), which implies QK(i) done.  The tensor pipe takes MMAs from both: one
      // warp's barrier polls and bookkeeping overlap the other's MMAs (one warp issuing both
      // left the pipe idle ~30 % of each tile).  A probe measured the same MMA throughput from
      // two issuing warps as from one.
      // (a phase seen complete by any lane is complete for all: only this warp's progress
      // can complete the next one)
      auto wait1 = [&](uint32_t bar_, uint32_t parity) -> bool {
        if (__any_sync(0xffffffffu, mbar_test(bar_, parity))) return true;
        return warp_bcast(mbar_wait(bar_, parity, abort_flag, prm.err));
      };
      Piece pc;
      uint32_t i = 0;
      bool ok = true;
      if (warp == LY::kQkWarp) {
        constexpr uint32_t idesc_qk = idesc_f8(128, LY::kTile, false, false);
        const uint64_t q_lat = smem_desc(sQ, 16, 1024, kSw128);
        const uint64_t q_rope = smem_desc(sQ + LY::kQRopeOff, 16, 512, kSw64);
        const uint64_t k_lat0 = smem_desc(sbase, 16, 1024, kSw128);
        const uint64_t k_rope0 = smem_desc(sbase + LY::kRopeOff, 16, 512, kSw64);
        int n_piece = 0;
        while (ok && iter.next(pc, &bad)) {
          const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
          for (int t = 0; t < nt && ok; ++t, ++i) {
            if (t == 0 && !wait1(mbase + LY::kQFull, n_piece & 1)) {
              ok = false;
              break;
            }
            const int stage = static_cast<int>(i % STAGES);
            if (!wait1(mbase + LY::kFull + 8 * stage, (i / STAGES) & 1)) {
              ok = false;
              break;
            }
            if (i > 0 && !wait1(mbase + LY::kSFree, (i - 1) & 1)) {
              ok = false;
              break;
            }
            // the stage was written by cp.async (generic proxy); the tensor core reads it
            // through the async proxy
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t ka = desc_at(k_lat0, stage * LY::kStageBytes);
            const uint64_t kr = desc_at(k_rope0, stage * LY::kStageBytes);
            const uint32_t d = tmem + LY::kSCol;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)   // latent columns, 32 per MMA: A = q, B = rows
              mma_f8_warp(d, desc_at(q_lat, (kk >> 2) * LY::kQLatBlock + (kk & 3) * 32),
                          desc_at(ka, (kk >> 2) * LY::kLatBlock + (kk & 3) * 32), idesc_qk,
                          kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              mma_f8_warp(d, desc_at(q_rope, kk * 32), desc_at(kr, kk * 32), idesc_qk, 1u);
            mma_commit_warp(mbase + LY::kSFull);
            if (t == nt - 1) mma_commit_warp(mbase + LY::kQEmpty);   // q may be overwritten
          }
          ++n_piece;
        }
        // Drain: all MMAs must complete before tensor memory is released.
        mma_commit_warp(mbase + LY::kDrain);
        if (lane == 0) mbar_wait_drain(mbase + LY::kDrain, 0);
      } else {
        constexpr uint32_t idesc_pv = idesc_f8_blockscaled(128, NG, true, false);
        const uint64_t v_lat0 = smem_desc(sbase, LY::kLatBlock, 1024, kSw128);
        // P, K-major without swizzle: 16-position chunks kPChunk apart (leading byte offset),
        // 8-row core matrices 128 bytes apart (stride byte offset)
        const uint64_t p_hi0 = smem_desc(sbase + LY::kPOff, LY::kPChunk, 128, kSwNone);
        const uint32_t sfa = tmem + LY::kSfA;
        const uint32_t sfh = tmem + LY::kSfHi;
        const uint32_t sfl = tmem + LY::kSfLo;
        while (ok && iter.next(pc, &bad)) {
          const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
          for (int t = 0; t < nt && ok; ++t, ++i) {
            if (!wait1(mbase + LY::kPFull + 8 * (i & 1), (i >> 1) & 1)) {
              ok = false;
              break;
            }
            const int stage = static_cast<int>(i % STAGES);
            tc_fence_after();
            const uint64_t va = desc_at(v_lat0, stage * LY::kStageBytes);
            const uint64_t ph = desc_at(p_hi0, (i & 1) * 2 * LY::kPPlane);
#pragma unroll
            for (int bk = 0; bk < 4; ++bk) {
              const uint32_t d = tmem + LY::kOBase + bk * NG;
#pragma unroll
              for (int kk = 0; kk < LY::kTile / 32; ++kk) {
                // A = V^T block bk (128 value columns x 32 positions); B = P (32 positions x
                // NG rows), hi plane at scale 1, lo plane at scale 2^-4
                const uint64_t a = desc_at(va, bk * LY::kLatBlock + kk * 32 * 128);
                mma_f8_scaled_warp(d, a, desc_at(ph, kk * 2 * LY::kPChunk), idesc_pv, sfa, sfh,
                                   (t == 0 && kk == 0) ? 0u : 1u);
                mma_f8_scaled_warp(d, a, desc_at(ph, LY::kPPlane + kk * 2 * LY::kPChunk),
                                   idesc_pv, sfa, sfl, 1u);
              }
            }
            // the stage (its QK finished before P(i) existed) and O's tile are released
            mma_commit_warp(mbase + LY::kEmpty + 8 * stage);
            mma_commit_warp(mbase + LY::kPv + 8 * (i & 1));
          }
        }
        mma_commit_warp(mbase + LY::kDrainPv);
        if (lane == 0) mbar_wait_drain(mbase + LY::kDrainPv, 0);
      }
      __syncwarp();
    }
  }
  if (bad && (threadIdx.x & 31) == 0) atomicOr(prm.err, kErrBadIndptr);
  tc_fence_before();
  __syncthreads();
  if (warp == LY::kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, LY::kTmemCols);
  }
}

}  // namespace pmla
