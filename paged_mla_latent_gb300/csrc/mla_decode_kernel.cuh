// Absorbed (latent) MLA decode over a page_size=1 FP8 cache on sm_103a.
//
// What it computes: "[Kimi-K3 MLA TP8] MLA performance" §2 (576-wide latent entry per
// token shared by every head, sm_scale = 1/sqrt(192)), §4.1 (fp8 q and cache, float32
// q_scale / kv_scale), §5.2 (page_size 1: one row id per position); softmax partials
// and their merge: "Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache" and §4 "MLA".
//
// One persistent CTA per SM walks the pieces the scheduler (mla_sched.cuh) gives it.
// Per tile of 128 cache positions (96 in the three-stage 32/48-row variants):
//   producer warps  : seven warps (0-3, 5-7), rows r = w + 7 j: load the row ids, then
//                     copy every row with 16-byte cp.async (one instruction per row of
//                     latent columns, lanes along the row; one per 8 rows of rope columns)
//                     straight into a 3- (or 2-) stage ring in the 128-byte (latent) /
//                     64-byte (rope) swizzled layouts the tensor core reads.  Positions
//                     past the piece and invalid row ids are zero-filled.  (Prefetching
//                     later tiles' rows into L2 measured slower: the extra requests cost
//                     more than the latency they hide.)  (A TMA tile::gather4 of
//                     128-byte boxes issues 5 requests per 4 rows and measured 2-4 TB/s on
//                     this access pattern; per-thread copies reach the random-row gather
//                     limit of ~5.3 TB/s.)
//   MMA warp        : (warp 4) S^T[pos, n] = K[pos, :] . Q[n, :]  (tcgen05 kind::f8f6f4,
//                     M = 128 positions, N = NG query rows, K = 576; FP32 in TMEM),
//                     then O^T[c, n] += V^T[c, pos] . P^T[pos, n] for the four 128-wide
//                     value blocks (A = the same cache rows read MN-major; N = 2 NG: the
//                     two P planes side by side).
//   softmax warps   : (one warpgroup per 16 query rows: warps 8-11, 12-15, 16-19) read
//                     their 16 columns of S^T from TMEM (one position per thread), scale, mask,
//                     online softmax in the exp2 domain with a lazily moved reference
//                     max, and write P (scaled by 2^6 relative to that max) as two FP8
//                     planes: hi = e4m3(p) and lo = e4m3(16 * (p - hi)), so P reaches
//                     the tensor core with ~2^-8 relative precision for weights down to
//                     2^-12 of the max while staying an FP8 x FP8 product.
//                     At the end of a piece they normalise O and write o / lse (or a
//                     normalised partial for the merge kernel).
#pragma once

#include <cuda_bf16.h>

#include "mla_sched.cuh"
#include "ptx.cuh"

namespace pmla {

struct DecodeParams {
  SchedParams sp;
  const uint8_t* kv;       // cache: slot s of page p at kv + p * page_pitch + s * kv_pitch
  int64_t kv_pitch;        // bytes between a page's slots (pages of one token: unused)
  int64_t page_pitch;      // bytes between pages (pages of 2^sp.log2_page tokens)
  const int32_t* kv_indices;
  int64_t kv_indices_len;
  int64_t n_kv_rows;       // pages in the cache
  int64_t n_q_rows;        // sum_T * H
  const float* q_scale;
  const float* kv_scale;
  float sm_scale;
  void* o;                 // (sum_T, H, 512), bf16 or fp32
  int o_fp32;
  int64_t o_stride_tok;    // elements
  int64_t o_stride_head;   // elements
  int o_vec16;             // o's base and strides allow 16-byte stores of 16-byte runs
  float* lse_out;          // (sum_T, H) or null
  float* part_o;           // (slots, NG, 512) normalised partial o (kv_scale applied)
  float* part_lse;         // (slots, NG) natural-log lse of each partial
  int64_t n_slots;
  int* err;
};

// Misc region offsets (bytes from kMiscOff).
enum : int {
  kMiscFull = 0,      // full[STAGES]   (8 B each, STAGES <= 4)
  kMiscEmpty = 32,    // empty[STAGES]
  kMiscSFull = 64,    // s_full[2]
  kMiscPFull = 80,    // p_full[2]
  kMiscPv = 96,       // pv_done[2]: PV of even / odd tiles (a single barrier would let a
                      // waiter two completions behind mistake an old phase for its own)
  kMiscQFull = 112,
  kMiscQEmpty = 120,
  kMiscDrain = 184,
  kMiscTmem = 128,    // u32 tensor memory base
  kMiscAbort = 132,   // int abort flag
  kMiscRowOff = 192,  // int64 row output offsets [NG] (NG <= 48 -> 384 bytes, to 576)
  kMiscRed = 640,     // float red[4][NG], then float scale / alpha [NG], then int lim[NG]
};

// Cache positions per pipeline tile.  The MMA's M is always 128 (TMEM lanes = positions);
// a three-stage ring of 128-position tiles does not fit in shared memory next to a 32- or
// 48-row q tile, one of 96-position tiles does.  Its QK reads 32 rows past each block
// (whatever the next block holds: finite or not, those logits are masked, their P is never
// written) and its PV runs three 32-position K steps.
constexpr int tile_positions(int NG, int STAGES) { return (STAGES >= 3 && NG >= 32) ? 96 : kTile; }

template <int NG, int STAGES>
struct DecodeLayout {
  static constexpr int kTile = tile_positions(NG, STAGES);
  static constexpr int kNPV = 2 * NG;                 // PV N: hi plane + lo plane
  static constexpr int kStageBytes = kTile * kD;      // 73,728 (128 positions)
  static constexpr int kLatBlock = kTile * 128;       // one 128-column latent block
  static constexpr int kRopeOff = 4 * kLatBlock;      // rope block inside a stage
  // P (2*NG rows x kTile positions) fits in the stage's rope block once QK has read it.
  static constexpr bool kPInRope = kNPV * kTile <= kTile * 64;
  static constexpr int kQOff = STAGES * kStageBytes;
  static constexpr int kQBytes = NG * kD;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kPBytes = kPInRope ? 0 : 2 * kNPV * kTile;
  // P tile: MN-major, no swizzle.  Position j's bytes for columns 16m .. 16m+15 are at
  // m * kPGroup + (j / 8) * 128 + (j % 8) * 16.
  static constexpr int kPGroup = kTile * 16;
  static constexpr int kRowsPerProducer = (kTile + 6) / 7;   // 19 (128) or 14 (96)
  static_assert(kTile % 32 == 0 && kTile <= 128, "tile must be whole PV K steps of one M");
  static_assert(kStageBytes % 1024 == 0 && kLatBlock % 1024 == 0, "swizzle atoms");
  static constexpr int kMiscOff = kPOff + kPBytes;
  static constexpr int kMiscBytes = (NG <= 16) ? 1024 : 3072;
  static constexpr int kMiscLim = kMiscRed + 5 * NG * 4;        // int causal limit [NG]
  // tile-max exchange of each softmax warpgroup (64 floats; one group uses red)
  static constexpr int kMiscXch = (kMiscLim + 4 * NG + 15) / 16 * 16;
  static_assert((NG <= 16 ? kMiscLim + 4 * NG : kMiscXch + 256 * (NG / 16)) <= kMiscBytes,
                "misc region overflow");
  static constexpr int kSmemBytes = kMiscOff + kMiscBytes;
  // Tensor memory columns: two S buffers, then four O blocks of kNPV columns.
  static constexpr int kSStride = (NG + 31) / 32 * 32;
  static constexpr int kOBase = 2 * kSStride;
  static constexpr int kTmemCols = (kOBase + 4 * kNPV <= 256) ? 256 : 512;
  static_assert(kOBase + 4 * kNPV <= 512, "tensor memory overflow");
  static_assert(kSmemBytes <= 232448, "shared memory overflow");
  static_assert(NG % 16 == 0 && NG <= 48, "group rows must be 16, 32 or 48");
  // Warps: 0-3 and 5-7 producers, 4 MMA issuer, then one softmax warpgroup per 16-column
  // chunk of the group's rows (warp 8 + 4 g + q: chunk g, TMEM lane quadrant q).
  static constexpr int kGroups = NG / 16;
  static constexpr int kThreads = 32 * (8 + 4 * kGroups);              // 384 / 512 / 640
  // Registers a thread is launched with (65,536 per SM, whole multiples of 8), and the
  // setmaxnreg split: the two producer/issuer warpgroups give registers back, the softmax
  // warpgroups take them.  The split must fit the launch allocation, or .inc waits forever.
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8 > 168 ? 168 : (65536 / kThreads) / 8 * 8;
  static constexpr int kRegsLow = NG == 16 ? 120 : (NG == 32 ? 104 : 80);
  static constexpr int kRegsHigh = NG == 16 ? 224 : (NG == 32 ? 152 : 104);
  static_assert(2 * kRegsLow + kGroups * kRegsHigh <= (2 + kGroups) * kLaunchRegs,
                "register split exceeds the launch allocation");
};


// Warpgroups 0 and 1 (producers + MMA issuer) give registers back with setmaxnreg.dec;
// the softmax warpgroups (one per 16-column chunk, see DecodeLayout) take them with .inc.
//   warps 0-3, 5-7 : producers (7 warps)      warp 4 : MMA issuer, TMEM owner
//   warps 8 + 4 g + q : softmax / epilogue of chunk g, TMEM lane quadrant q
constexpr int kProducerWarps = 7;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kMmaWarp = 4;
constexpr int kSoftmaxWarp0 = 8;
constexpr int kSoftmaxThread0 = 32 * kSoftmaxWarp0;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// P in FP8.  Each column keeps m = (reference max) - kPShift, and a logit x (log2 units)
// becomes p = 2^(x - m): the column's probabilities scaled by 2^kPShift relative to the
// reference.  The reference moves only when a logit exceeds it by more than kHeadroom, so
// O is rescaled rarely and p <= 2^kMoveAt = 256 (< 448, the e4m3 maximum).  p reaches the
// tensor core as two planes, hi = e4m3(p) and lo = e4m3(kLoScale (p - hi)): e4m3 rounds p
// within p / 16, so lo <= p <= 256 also fits, and hi + lo / kLoScale carries ~2^-8
// relative precision for every p >= 2^-6, i.e. for weights down to 2^-12 of the reference
// (a sink far above a large uniform bulk keeps the bulk's mass).  The row sum l accumulates
// the same scaled p, so o = (O_hi + O_lo / kLoScale) / l and lse = (m + log2 l) ln 2 need
// no correction for the scale.
constexpr float kPShift = 6.0f;
constexpr float kHeadroom = 2.0f;
constexpr float kMoveAt = kHeadroom + kPShift;
constexpr float kLoScale = 16.0f;
constexpr uint32_t kLoScaleF16x2 = 0x4C004C00u;   // kLoScale as two f16
// Initial reference max: finite, so that p = 2^(x - ref) needs no special case (masked
// logits are -inf and give 0) and the first tile always moves it (x - m > kMoveAt).
constexpr float kRefInit = -1.0e30f;

// Warp-wide reduction of 16 per-lane column values v[0..15] (sum or max): four halving
// exchanges leave lane l with column col16(l) reduced over the lanes sharing bits 1..4
// of l, a fifth exchange completes it.  16 shuffles instead of 16 x 5.
__device__ __forceinline__ int col16(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}
template <bool kMax>
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int half = 8, m = 16; half >= 1; half >>= 1, m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = up ? v[j] : v[j + half];
      const float keep = up ? v[j + half] : v[j];
      const float got = __shfl_xor_sync(0xffffffffu, send, m);
      v[j] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  const float got = __shfl_xor_sync(0xffffffffu, v[0], 1);
  return kMax ? fmaxf(v[0], got) : v[0] + got;
}

// In-register transpose of W x W blocks among groups of W lanes (W = 4 or 8): lane i of a
// group holds a[j] = element (i, j); afterwards it holds a[j] = element (j, i).
template <int W>
__device__ __forceinline__ void lane_transpose(float* a, int lane) {
#pragma unroll
  for (int m = W / 2; m >= 1; m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      if ((j & m) == 0) {
        const float send = up ? a[j] : a[j | m];
        const float got = __shfl_xor_sync(0xffffffffu, send, m);
        if (up)
          a[j] = got;
        else
          a[j | m] = got;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// q rows [qrow, qrow + NG) of the group into shared memory: one TMA tile load per
// 128-byte latent block and one for the rope block, completing on `bar`.  Rows past the
// unit's real rows belong to other requests (or are out of range and read zeros); their
// columns are discarded.
template <int NG>
__device__ __forceinline__ void issue_q_load(uint32_t sQ, const CUtensorMap* lat,
                                             const CUtensorMap* rope, int qrow, uint32_t bar) {
  mbar_arrive_expect_tx(bar, NG * kD);
#pragma unroll
  for (int c = 0; c < 4; ++c) tma_load_2d(sQ + c * NG * 128, lat, c * 128, qrow, bar);
  tma_load_2d(sQ + 4 * NG * 128, rope, 512, qrow, bar);
}

// MODE: the schedule (kSchedWhole for a plain decode, kSchedCascade for the shared-prefix
// cascade), fixed at compile time.
template <int NG, int STAGES, int MODE>
__global__ void __launch_bounds__(DecodeLayout<NG, STAGES>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q_lat,
                      const __grid_constant__ CUtensorMap tm_q_rope, const DecodeParams prm) {
  using LY = DecodeLayout<NG, STAGES>;
  constexpr int NPV = LY::kNPV;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t mbase = sbase + LY::kMiscOff;
  uint8_t* misc = smem + LY::kMiscOff;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc + kMiscTmem);
  const uint32_t sQ = sbase + LY::kQOff;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + kMiscAbort);
  float* red = reinterpret_cast<float*>(misc + kMiscRed);

  if ((sbase & 1023u) != 0) {   // the swizzled layouts need a 1024-byte aligned window
    if (threadIdx.x == 0) atomicOr(prm.err, kErrMisaligned);
    return;
  }

  if (threadIdx.x == 64) {   // descriptors of the q loads, fetched while the schedule is read
    prefetch_tensormap(&tm_q_lat);
    prefetch_tensormap(&tm_q_rope);
  }
  // The schedule reads kv_indptr and then qo_indptr; fetch both arrays' first lines at
  // once so that the second read does not wait for a second trip to memory.
  if (threadIdx.x < 64) {
    const int i = 32 * (threadIdx.x >> 1);
    if (i <= prm.sp.B) prefetch_l1((threadIdx.x & 1) ? prm.sp.qo_indptr + i : prm.sp.kv_indptr + i);
  }
  PieceIterT<MODE> iter;
  iter.init(prm.sp, blockIdx.x);
  int first_qrow;   // q row of the first piece's group (its q load starts in the set-up)
  {
    Piece pc;
    int bad = 0;
    if (!iter.next(pc, &bad)) {    // no work for this CTA (uniform across the block)
      if (bad && threadIdx.x == 0) atomicOr(prm.err, kErrBadIndptr);
      return;
    }
    iter.hold(pc);                 // every role starts from this piece
    first_qrow = pc.qo0 * prm.sp.H + pc.g * NG;
    // the first tile's row ids: their fetch overlaps the set-up below
    if (threadIdx.x < LY::kTile / 32) {
      const int64_t gi = pc.kv0 + ((pc.j0 + 32 * threadIdx.x) >> prm.sp.log2_page);
      if (gi >= 0 && gi < prm.kv_indices_len) prefetch_l1(prm.kv_indices + gi);
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(mbase + kMiscFull + 8 * s, kProducerThreads);   // one cp.async arrival per producer thread
      mbar_init(mbase + kMiscEmpty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(mbase + kMiscSFull + 8 * s, 1);
      mbar_init(mbase + kMiscPFull + 8 * s, 4 * LY::kGroups);   // every softmax warp
    }
    mbar_init(mbase + kMiscPv, 1);
    mbar_init(mbase + kMiscPv + 8, 1);
    mbar_init(mbase + kMiscQFull, 1);
    mbar_init(mbase + kMiscQEmpty, 1);
    mbar_init(mbase + kMiscDrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    issue_q_load<NG>(sQ, &tm_q_lat, &tm_q_rope, first_qrow, mbase + kMiscQFull);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(misc + kMiscTmem), LY::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Let the merge grid (launched with programmatic serialization) get scheduled; it
  // waits for this grid's completion before reading anything it wrote.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp >= kSoftmaxWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(LY::kRegsHigh));
    // ===================================================== softmax + epilogue
    // Warpgroup g owns columns (query rows of the group) c0 = 16 g .. c0 + 15, warp q of it
    // TMEM lane quadrant q (positions 32 q .. 32 q + 31).  The warpgroups share only the
    // tile handshakes (S full, P full, PV done); each votes, exchanges tile maxima, reduces
    // and writes its rows out on its own named barrier, so they run side by side.
    // They read their first piece again (from memory: off their critical path, they wait
    // for the first tile's logits) and so keep no held piece in registers.
    iter.init(prm.sp, blockIdx.x);
    const int grp = (warp - kSoftmaxWarp0) >> 2;
    const int bar_g = 1 + grp;               // named barrier of this warpgroup (128 threads)
    const int c0 = 16 * grp;                 // its first column
    const int q4 = warp & 3;                 // TMEM lane quadrant this warp may access
    const int prow = 32 * q4 + lane;         // position within the tile == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const float kv_scale = *prm.kv_scale;
    const float scale_log2 = prm.sm_scale * (*prm.q_scale) * kv_scale * kLog2e;
    const int H = prm.sp.H;
    // P is stored MN-major without swizzle (see the PV descriptor): this position's 16
    // bytes of columns 16m .. 16m+15 sit at pofs + m * LY::kPGroup.
    const uint32_t pofs = (prow >> 3) * 128 + (prow & 7) * 16;
    float* s_alpha = red + 4 * NG + c0;      // this chunk's rescale factors [16]
    float* xch = LY::kGroups == 1 ? red
                                  : reinterpret_cast<float*>(misc + LY::kMiscXch) + 64 * grp;
    int* s_lim = reinterpret_cast<int*>(misc + LY::kMiscLim);   // 16-row kernel only
    constexpr int kCh = NG / 16;

    uint32_t it_g = 0;
    Piece pc;
    float m_ref[16];   // reference max - kPShift, per column of the chunk
    float l_acc[16];
    while (iter.next(pc, &bad)) {
      const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
      // A chunk past the unit's real rows (a 12-row unit in a 48-row tile) is skipped: its P
      // columns only feed O columns that are never written out.
      const bool live = c0 < pc.rows;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        m_ref[k] = kRefInit;
        l_acc[k] = 0.f;
      }
      const int causal_from = pc.cfrom;   // positions beyond this need the causal test
      if constexpr (NG == 16) {
        // draft t of this group's row n sees positions <= causal_from + t (16-row kernel:
        // one limit per column in shared memory, see the masks below)
        if (prow < 16) s_lim[c0 + prow] = causal_from + (pc.g * NG + c0 + prow) / H;
        bar_sync(bar_g, 128);
      }
      for (int t = 0; t < nt; ++t, ++it_g) {
        const int sb = it_g & 1;
        mbar_wait(mbase + kMiscSFull + 8 * sb, (it_g >> 1) & 1, abort_flag, prm.err);
        tc_fence_after();
        if (live) {
          const int pos = pc.j0 + t * LY::kTile + prow;
          // (lanes past a 96-position tile hold don't-care logits and write no P)
          const bool in_piece = prow < LY::kTile && pos < pc.j1;
          // Scaled logits (log2 units) with masks: past the piece or beyond the draft's
          // causal limit -> -inf; padding rows -> 0 (finite, discarded).
          const int stage = static_cast<int>(it_g % STAGES);
          // P tile: this position's 16-byte vectors (see LY::kPGroup)
          uint8_t* pb = (LY::kPInRope ? smem + stage * LY::kStageBytes + LY::kRopeOff
                                      : smem + LY::kPOff + sb * NPV * LY::kTile) + pofs;
          float xs[16];
          tmem_ld16(tl + sb * LY::kSStride + c0, xs);
          tmem_wait_ld();
          float dmax = -INFINITY;
          if constexpr (NG == 16) {
            // One limit per column, read from shared memory.  (The per-tile cut below, and
            // even the row bound held as (rows - c0) across the tile loop, measured 4 %
            // slower on the 16-row kernel's calls, with fewer instructions executed and more
            // instruction-fetch stalls; the cause was not found.)
            const bool causal = in_piece && pos > causal_from;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float v = in_piece ? xs[k] * scale_log2 : -INFINITY;
              if (causal && pos > s_lim[c0 + k]) v = -INFINITY;
              xs[k] = (c0 + k >= pc.rows) ? 0.f : v;
              dmax = fmaxf(dmax, xs[k] - m_ref[k]);
            }
          } else if (prow >= LY::kTile) {
            // lanes past a 96-position tile (a whole warp) hold no position
#pragma unroll
            for (int k = 0; k < 16; ++k) xs[k] = -INFINITY;
          } else {
            // Row r = pc.g * NG + c0 + k of the group is draft r / H, which sees positions
            // <= causal_from + r / H: at position pos the columns beyond their drafts' limits
            // are the prefix k < (pos - causal_from) * H - (pc.g * NG + c0) of the chunk (none
            // at or before causal_from).  One cut per tile, and no masks at all for interior
            // positions with 16 real rows: the softmax warps share their schedulers with the
            // producer and MMA warps, and their time per tile follows their instruction count
            // (a per-column limit read from shared memory cost ~0.3 us a tile in the
            // shared-prefix call).
            const int rows_left = pc.rows - c0;   // columns k >= rows_left are padding rows
            const int64_t cut = static_cast<int64_t>(pos - causal_from) * H - (pc.g * NG + c0);
            const int kcut = static_cast<int>(cut < 0 ? 0 : (cut > 16 ? 16 : cut));
            if (in_piece && kcut == 0 && rows_left >= 16) {
#pragma unroll
              for (int k = 0; k < 16; ++k) xs[k] *= scale_log2;
            } else if (in_piece && kcut == 0) {
#pragma unroll
              for (int k = 0; k < 16; ++k) xs[k] = k < rows_left ? xs[k] * scale_log2 : 0.f;
            } else {
              const int kc = in_piece ? kcut : 16;
#pragma unroll
              for (int k = 0; k < 16; ++k)
                xs[k] = k < rows_left ? (k < kc ? -INFINITY : xs[k] * scale_log2) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) dmax = fmaxf(dmax, xs[k] - m_ref[k]);
          }
          if (bar_red_or(bar_g, 128, dmax > kMoveAt)) {
            // rare: move these columns' reference to their tile maxima
            {
              float v[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] = xs[k];
              const float wmax = reduce_scatter16<true>(v, lane);
              if ((lane & 1) == 0) xch[col16(lane) * 4 + q4] = wmax;
            }
            bar_sync(bar_g, 128);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float4 r4 = *reinterpret_cast<const float4*>(xch + 4 * k);
              const float tmax = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
              const float m_new = fmaxf(m_ref[k], tmax - kPShift);
              const float alpha = ex2_approx(m_ref[k] - m_new);   // 0 from the initial reference
              l_acc[k] *= alpha;
              m_ref[k] = m_new;
              if (prow == 0) s_alpha[k] = alpha;
            }
            bar_sync(bar_g, 128);
            if (t > 0) {
              // O holds this piece's earlier tiles: wait for the last PV, then rescale the
              // chunk's hi and lo columns in the four value blocks
              mbar_wait(mbase + kMiscPv + 8 * ((it_g - 1) & 1), ((it_g - 1) >> 1) & 1, abort_flag,
                        prm.err);
              tc_fence_after();
#pragma unroll 1
              for (int bp = 0; bp < 8; ++bp) {
                float v[16];
                const uint32_t a = tl + LY::kOBase + (bp >> 1) * NPV + (bp & 1) * NG + c0;
                tmem_ld16(a, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] *= s_alpha[k];
                tmem_st16(a, v);
              }
              tmem_wait_st();
            }
          }
          // scaled probabilities (<= 2^kMoveAt), split into two FP8 planes:
          // hi = e4m3(p), lo = e4m3(kLoScale (p - hi)), the residual taken in f16x2
          // (positions past a 96-position tile hold no P: their weights are 0 and their
          // lanes skip the conversion)
          if (LY::kTile == 128 || prow < LY::kTile) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              const float p0 = ex2_approx(xs[k] - m_ref[k]);
              const float p1 = ex2_approx(xs[k + 1] - m_ref[k + 1]);
              l_acc[k] += p0;
              l_acc[k + 1] += p1;
              const uint32_t p16 = f32x2_to_f16x2(p1, p0);          // low half: p0
              const uint32_t hi = f16x2_to_e4m3x2(p16);             // byte 0: p0, byte 1: p1
              const uint32_t r16 = f16x2_mul(f16x2_sub(p16, e4m3x2_to_f16x2(hi)), kLoScaleF16x2);
              const uint32_t lo = f16x2_to_e4m3x2(r16);              // kLoScale (p - hi)
              if ((k & 2) == 0) {
                hw[k >> 2] = hi;
                lw[k >> 2] = lo;
              } else {
                hw[k >> 2] |= hi << 16;
                lw[k >> 2] |= lo << 16;
              }
            }
            *reinterpret_cast<uint4*>(pb + grp * LY::kPGroup) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(pb + (kCh + grp) * LY::kPGroup) =
                make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(mbase + kMiscPFull + 8 * sb);
      }
      // ------------------------------------------------ piece epilogue (after its last
      // tile's P was handed to the MMA issuer; kept out of the tile loop)
      {
        const uint32_t it_last = it_g - 1;
        // The row sums and the per-row set-up need only the softmax state: they run while
        // the piece's last PV is still in the tensor pipe; the output waits for it.
        if (live) {
          float v[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = l_acc[k];
          const float wsum = reduce_scatter16<false>(v, lane);
          if ((lane & 1) == 0) red[q4 * NG + c0 + col16(lane)] = wsum;
        }
        bar_sync(bar_g, 128);
        // one thread per row: normaliser, lse and output offset of that row
        float* s_scale = red + 4 * NG;                                   // [NG]
        int64_t* s_off = reinterpret_cast<int64_t*>(misc + kMiscRowOff);  // [NG]
        const bool direct = pc.direct;
        const bool slot_ok = direct || (pc.slot >= 0 && pc.slot < prm.n_slots);
        if (live && prow < 16) {
          const int n = c0 + prow;
          const float l = (red[n] + red[NG + n]) + (red[2 * NG + n] + red[3 * NG + n]);
          float m = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) m = (k == prow) ? m_ref[k] : m;
          const float lse = (l > 0.f) ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
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
        bar_sync(bar_g, 128);
        if (live) {
          mbar_wait(mbase + kMiscPv + 8 * (it_last & 1), (it_last >> 1) & 1, abort_flag, prm.err);
          tc_fence_after();
          // normalised output.  TMEM lane = value column: a warp holds 32 adjacent columns
          // of every row.  Lanes exchange values (in-register transposes) so that each
          // writes 16 contiguous bytes of one row: 8 bf16 columns (rows i, i + 8 of the
          // chunk for lane i of 8) or 4 fp32 columns (rows i, i + 4, i + 8, i + 12 for lane
          // i of 4).  Scalar stores when o's layout does not allow 16-byte stores.
          const bool to_bf16 = direct && !prm.o_fp32;
          const bool vec = !direct || prm.o_vec16;
          float* fdst = direct ? reinterpret_cast<float*>(prm.o) : prm.part_o;
          __nv_bfloat16* hdst = reinterpret_cast<__nv_bfloat16*>(prm.o);
          // the rows' scales and this lane's output rows, read once for the four blocks
          float scl[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) scl[k] = s_scale[c0 + k];
          int64_t offq[4];
#pragma unroll
          for (int g = 0; g < 4; ++g)
            offq[g] = s_off[c0 + (to_bf16 ? 8 * (g & 1) + (lane & 7) : 4 * g + (lane & 3))];
          #pragma unroll 1
          for (int bk = 0; bk < 4; ++bk) {
            float hi[16], lo[16];
            tmem_ld16(tl + LY::kOBase + bk * NPV + c0, hi);
            tmem_ld16(tl + LY::kOBase + bk * NPV + NG + c0, lo);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) hi[k] = (hi[k] + lo[k] * (1.0f / kLoScale)) * scl[k];
            const int cw = bk * 128 + 32 * q4;   // first column of this warp
            if (!vec) {
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const int64_t off = s_off[c0 + k];
                if (off < 0) continue;
                if (to_bf16)
                  hdst[off + cw + lane] = __float2bfloat16_rn(hi[k]);
                else
                  fdst[off + cw + lane] = hi[k];
              }
            } else if (to_bf16) {
              lane_transpose<8>(hi, lane);
              lane_transpose<8>(hi + 8, lane);
              const int cs = cw + 8 * (lane >> 3);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int64_t off = offq[h];
                if (off >= 0) {
                  const float* a = hi + 8 * h;
                  *reinterpret_cast<uint4*>(hdst + off + cs) =
                      make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                 pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
                }
              }
            } else {
#pragma unroll
              for (int g = 0; g < 4; ++g) lane_transpose<4>(hi + 4 * g, lane);
              const int cs = cw + 4 * (lane >> 2);
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int64_t off = offq[g];
                if (off >= 0)
                  *reinterpret_cast<float4*>(fdst + off + cs) =
                      make_float4(hi[4 * g], hi[4 * g + 1], hi[4 * g + 2], hi[4 * g + 3]);
              }
            }
          }
        }
        bar_sync(bar_g, 128);   // s_off / s_scale are rewritten by the next piece
        tc_fence_before();
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LY::kRegsLow));
    if (warp != kMmaWarp) {
      // ===================================================== producers (7 warps)
      const int pw = warp < kMmaWarp ? warp : warp - 1;   // producer index 0..6
      uint32_t it_g = 0;
      int n_piece = 0;
      int q_loads = 0;
      bool aborted = false;
      Piece pc;
      const uint8_t* kv = prm.kv;
      // Position pos of a request lies in its page pos >> log2_page, slot pos & (size - 1);
      // the row's bytes start at kv + page * page_pitch + slot * kv_pitch.  Each lane turns
      // its row into that byte offset once; the copy loops only shuffle it.
      const int lg = prm.sp.log2_page;
      const int smask = (1 << lg) - 1;
      const int64_t ppitch = prm.page_pitch;
      const int64_t spitch = prm.kv_pitch;
      // Producer pw copies tile rows r = pw + 7 j (j < rows_w); lane j loads row j's id.
      const int rows_w = (LY::kTile - pw + kProducerWarps - 1) / kProducerWarps;   // 19 / 18 (14 / 13)
      while (!aborted && iter.next(pc, &bad)) {
        const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
        if (warp == 0 && lane == 0) {
          // q rows of this piece, once the previous piece's QK has released the buffer
          // (the first piece's load was issued during the set-up)
          if (n_piece == 0) {
            ++q_loads;
          } else if (!mbar_wait(mbase + kMiscQEmpty, (n_piece - 1) & 1, abort_flag, prm.err)) {
            aborted = true;
          } else {
            issue_q_load<NG>(sQ, &tm_q_lat, &tm_q_rope, pc.qo0 * prm.sp.H + pc.g * NG,
                             mbase + kMiscQFull);
            ++q_loads;
          }
        }
        aborted = __shfl_sync(0xffffffffu, aborted ? 1 : 0, 0) != 0;
        if (aborted) break;
        const int64_t kvbase = pc.kv0;
        // byte offset of row j of this warp in tile t (-1: past the piece or invalid)
        auto load_row = [&](int t, int j) -> int64_t {
          if (j >= rows_w) return -1;
          const int pos = pc.j0 + t * LY::kTile + pw + kProducerWarps * j;
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
          // rows past the piece or invalid copy nothing: a bit mask by row, offsets clamped
          const uint32_t vmask = __ballot_sync(0xffffffffu, nxt >= 0);
          const int64_t rid = nxt >= 0 ? nxt : 0;
          if (t + 1 < nt) nxt = load_row(t + 1, lane);   // next tile's row ids overlap the wait
          if (t + 2 < nt && lane < rows_w) {   // and the one after is fetched into L1
            const int64_t gi = kvbase + ((pc.j0 + (t + 2) * LY::kTile + pw + kProducerWarps * lane) >> lg);
            if (gi >= 0 && gi < prm.kv_indices_len &&
                pc.j0 + (t + 2) * LY::kTile + pw + kProducerWarps * lane < pc.j1)
              prefetch_l1(prm.kv_indices + gi);
          }
          // Whole-request schedules take every row's offset into every lane before the wait,
          // so that the copy loop issues its copies back to back: 1-2.5 % faster calls on
          // the plain, mtp and 96-head workloads, 2 % slower on 128-token pages.  The
          // shared-prefix schedules measured ~1 % slower that way and keep the shuffle in the
          // loop.  (Compiling both loops into the whole-request kernel, chosen at run time by
          // the page size, made every workload slower than either.)
          constexpr bool kHoist = MODE == kSchedWhole;
          int64_t offs[kHoist ? LY::kRowsPerProducer : 1];
          if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < LY::kRowsPerProducer; ++j)
              offs[j] = __shfl_sync(0xffffffffu, rid, j);
          }
          if (use > 0 &&
              !mbar_wait(mbase + kMiscEmpty + 8 * stage, (use - 1) & 1, abort_flag, prm.err)) {
            aborted = true;
            break;
          }
          const uint32_t st = sbase + stage * LY::kStageBytes;
          // latent columns: one row per instruction, lane = 16-byte chunk (coalesced 512 B)
          const uint32_t blk = (lane >> 3) * LY::kLatBlock;
          const uint32_t chunk = lane & 7;
          if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < LY::kRowsPerProducer; ++j) {
              if (j < rows_w) {
                const int r = pw + kProducerWarps * j;
                const uint32_t dst = st + blk + r * 128 + ((chunk ^ (r & 7)) << 4);
                cp_async_16(dst, kv + offs[j] + 16 * lane, ((vmask >> j) & 1u) << 4);
              }
            }
          } else {
#pragma unroll 4
            for (int j = 0; j < rows_w; ++j) {
              const int r = pw + kProducerWarps * j;
              const int64_t off = __shfl_sync(0xffffffffu, rid, j);
              const uint32_t dst = st + blk + r * 128 + ((chunk ^ (r & 7)) << 4);
              cp_async_16(dst, kv + off + 16 * lane, ((vmask >> j) & 1u) << 4);
            }
          }
          // rope columns: 8 rows x 4 chunks per instruction
#pragma unroll
          for (int m = 0; m < (LY::kRowsPerProducer + 7) / 8; ++m) {
            const int j = 8 * m + (lane >> 2);
            const int c = lane & 3;
            const int64_t off = __shfl_sync(0xffffffffu, rid, j);
            if (j < rows_w) {
              const int r = pw + kProducerWarps * j;
              const uint32_t dst = st + LY::kRopeOff + r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
              cp_async_16(dst, kv + off + 512 + 16 * c, ((vmask >> j) & 1u) << 4);
            }
          }
          cp_async_arrive_noinc(mbase + kMiscFull + 8 * stage);
        }
        ++n_piece;
      }
      // Drain: every copy this warp issued must land before the CTA may exit.
      cp_async_wait_all();
      if (warp == 0 && lane == 0 && q_loads > 0)
        mbar_wait_drain(mbase + kMiscQFull, (q_loads - 1) & 1);
      __syncwarp();
    } else {
      // ===================================================== MMA issuer (one warp)
      // The whole warp runs the issue loop, so that the descriptors are warp-uniform values,
      // and one elected lane issues each MMA and commit (mma_f8_warp).  Every lane waits on
      // a barrier together (each wait is bounded); lane 0's outcome decides for the warp, so
      // its control flow stays uniform.  (A wait by lane 0 alone while the other lanes sat
      // in the broadcast made the first MMAs of a CTA take ~5 us.)
      {
        auto wait1 = [&](uint32_t bar_, uint32_t parity) -> bool {
          return warp_bcast(mbar_wait(bar_, parity, abort_flag, prm.err));
        };
        auto test1 = [&](uint32_t bar_, uint32_t parity) -> bool {
          bool r = false;
          if (lane == 0) r = mbar_test(bar_, parity);
          return warp_bcast(r);
        };
        constexpr uint32_t idesc_qk = idesc_f8(128, NG, false, false);
        constexpr uint32_t idesc_pv = idesc_f8(128, NPV, true, true);
        int n_piece = 0;
        Piece pc;
        // Descriptors are built once, for stage 0, P buffer 0 and the q tile; every MMA's
        // operand is one of them moved by a compile-time byte offset (desc_at: one 32-bit
        // add), plus a stage or buffer offset once per tile.  The issuing warp shares its
        // sub-partition with producer and softmax warps, so the instructions between MMAs
        // count: building both descriptors from addresses for every MMA cost 2-4 % of the
        // call time on every workload.
        const uint64_t k_lat0 = smem_desc(sbase, 16, 1024, kSw128);              // K, latent
        const uint64_t k_rope0 = smem_desc(sbase + LY::kRopeOff, 16, 512, kSw64);  // K, rope
        const uint64_t v_lat0 = smem_desc(sbase, LY::kLatBlock, 1024, kSw128);    // V^T
        const uint64_t q_lat = smem_desc(sQ, 16, 1024, kSw128);
        const uint64_t q_rope = smem_desc(sQ + 4 * NG * 128, 16, 512, kSw64);
        // P, MN-major without swizzle: 32 positions (K) in 8-position core matrices of 128
        // bytes, 128 bytes apart (leading byte offset); NPV columns (MN) in groups of 16,
        // LY::kPGroup apart (stride byte offset)
        const uint64_t p0 = smem_desc(LY::kPInRope ? sbase + LY::kRopeOff : sbase + LY::kPOff, 128,
                                      LY::kPGroup, kSwNone);
        auto issue_pv = [&](uint32_t i, bool first_of_piece) {
          const int sb = i & 1;
          const int stage = static_cast<int>(i % STAGES);
          tc_fence_after();
          const uint64_t va = desc_at(v_lat0, stage * LY::kStageBytes);
          const uint64_t pb = desc_at(p0, LY::kPInRope ? stage * LY::kStageBytes : sb * NPV * LY::kTile);
#pragma unroll
          for (int bk = 0; bk < 4; ++bk) {
            const uint32_t d = tmem + LY::kOBase + bk * NPV;
#pragma unroll
            for (int kk = 0; kk < LY::kTile / 32; ++kk) {
              // A = V^T block bk: 128 value columns (MN, contiguous) x 32 positions (K);
              // B = P: 32 positions (K) x NPV columns
              mma_f8_warp(d, desc_at(va, bk * LY::kLatBlock + kk * 32 * 128),
                          desc_at(pb, kk * 4 * 128), idesc_pv,
                          (first_of_piece && kk == 0) ? 0u : 1u);
            }
          }
          mma_commit_warp(mbase + kMiscEmpty + 8 * stage);
          mma_commit_warp(mbase + kMiscPv + 8 * (i & 1));
        };
        auto issue_qk = [&](uint32_t i) {
          const int stage = static_cast<int>(i % STAGES);
          // the stage was written by cp.async (generic proxy); the tensor core reads it
          // through the async proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint64_t ka = desc_at(k_lat0, stage * LY::kStageBytes);
          const uint64_t kr = desc_at(k_rope0, stage * LY::kStageBytes);
          const uint32_t d = tmem + (i & 1) * LY::kSStride;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)   // latent columns 0..511, 32 per MMA
            mma_f8_warp(d, desc_at(ka, (kk >> 2) * LY::kLatBlock + (kk & 3) * 32),
                        desc_at(q_lat, (kk >> 2) * NG * 128 + (kk & 3) * 32), idesc_qk,
                        kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)    // rope columns 512..575
            mma_f8_warp(d, desc_at(kr, kk * 32), desc_at(q_rope, kk * 32), idesc_qk, 1u);
          mma_commit_warp(mbase + kMiscSFull + 8 * (i & 1));
        };
        if constexpr (STAGES >= 3) {
          // Issue order: QK(0), QK(1), PV(0), QK(2), PV(1), ... (CTA-wide tile numbers): QK
          // runs one tile ahead of PV, so the tensor pipe computes the next logits while the
          // softmax warps work, and QK(i+1) reuses the S buffer of tile i-1 only after PV(i-1)
          // was issued, i.e. after its softmax finished.  Each step waits (bounded) for its
          // own inputs: the stage's rows (and the piece's q rows) for QK, P for PV.
          uint32_t i = 0;              // next tile to QK
          bool pend = false;           // the PV of tile pend_j is still to be issued
          uint32_t pend_j = 0;
          bool pend_first = false;     // ... and that tile is its piece's first
          bool ok = true;
          auto pv_step = [&]() {
            const uint32_t j = pend_j;
            if (!wait1(mbase + kMiscPFull + 8 * (j & 1), (j >> 1) & 1)) {
              ok = false;
              return;
            }
            issue_pv(j, pend_first);
            pend = false;
          };
          while (ok && iter.next(pc, &bad)) {
            const int nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
            for (int t = 0; t < nt && ok; ++t) {
              if (t == 0 && !wait1(mbase + kMiscQFull, n_piece & 1)) {
                ok = false;
                break;
              }
              const int stage = static_cast<int>(i % STAGES);
              if (!wait1(mbase + kMiscFull + 8 * stage, (i / STAGES) & 1)) {
                ok = false;
                break;
              }
              issue_qk(i);
              if (t == nt - 1) mma_commit_warp(mbase + kMiscQEmpty);   // the producers may overwrite q
              if (pend) pv_step();
              pend = true;
              pend_j = i;
              pend_first = (t == 0);
              ++i;
            }
            ++n_piece;
          }
          if (ok && pend) pv_step();
        } else {
          // (Rings of two stages; no current instantiation.)  With two stages, QK(i+1)
          // needs the stage PV(i-1) is about to release: a fixed order would idle the tensor
          // pipe on that reload, so issue whichever step is ready first.
          // Issue loop.  QK of tile q needs its cache rows (full), the piece's q rows and a
          // free S buffer (PV of tile q-2 issued); PV of tile p needs P (p_full).  Whichever
          // is ready goes first, PV preferred: it releases a ring stage to the producers.
          bool pv_first[2] = {false, false};
          uint32_t q_next = 0, p_next = 0;   // next tile for QK / PV (CTA-wide numbering)
          bool have_piece = false, q_ready = false;
          int nt = 0, t_in = 0;
          unsigned long long idle_since = 0;
          while (true) {
            while (!have_piece || t_in >= nt) {
              if (!iter.next(pc, &bad)) {
                have_piece = false;
                break;
              }
              have_piece = true;
              nt = (pc.j1 - pc.j0 + LY::kTile - 1) / LY::kTile;
              t_in = 0;
              q_ready = false;
            }
            if (!have_piece && p_next == q_next) break;   // everything issued
            bool progressed = false;
            if (p_next < q_next && test1(mbase + kMiscPFull + 8 * (p_next & 1), (p_next >> 1) & 1)) {
              issue_pv(p_next, pv_first[p_next & 1]);
              ++p_next;
              progressed = true;
            } else if (have_piece && q_next <= p_next + 1) {
              if (t_in == 0 && !q_ready) q_ready = test1(mbase + kMiscQFull, n_piece & 1);
              const int stage = static_cast<int>(q_next % STAGES);
              if ((t_in > 0 || q_ready) &&
                  test1(mbase + kMiscFull + 8 * stage, (q_next / STAGES) & 1)) {
                issue_qk(q_next);
                pv_first[q_next & 1] = (t_in == 0);
                if (t_in == nt - 1) {
                  mma_commit_warp(mbase + kMiscQEmpty);   // the producers may overwrite q rows
                  ++n_piece;
                }
                ++q_next;
                ++t_in;
                progressed = true;
              }
            }
            if (progressed) {
              idle_since = 0;
            } else {
              if (warp_bcast(*abort_flag != 0)) break;
              const unsigned long long now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
              if (idle_since == 0) {
                idle_since = now;
              } else if (now - idle_since > kWaitLimitNs) {
                if (lane == 0) {
                  *abort_flag = 1;
                  atomicOr(prm.err, kErrTimeout);
                }
                break;
              }
            }
          }
        }
        // Drain: all MMAs must complete before tensor memory is released.
        mma_commit_warp(mbase + kMiscDrain);
        if (lane == 0) mbar_wait_drain(mbase + kMiscDrain, 0);
      }
      __syncwarp();
    }
  }
  if (bad && (threadIdx.x & 31) == 0) atomicOr(prm.err, kErrBadIndptr);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, LY::kTmemCols);
  }
}

}  // namespace pmla
