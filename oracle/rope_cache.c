/*
 * FP32/FP8 oracle of the step before the decode -- TEST INFRASTRUCTURE ONLY (the CUDA
 * library never links or calls it; it shares no code with the library).
 *
 * "[Kimi-K3 MLA TP8] MLA performance" §3 "Entry point": the decode's q comes out of a
 * fused step that rotates the rope part of q, concatenates it after the 512 latent
 * columns, and writes the step's new latent cache entry into the cache the decode reads;
 * §2 "K3 MLA geometry": an entry is 576 wide, 512 latent + 64 rope (qk_rope_head_dim 64);
 * §4.1: q and the cache are float8_e4m3fn with float32 per-tensor scales q_scale and
 * kv_scale.  The pages do not print the rotation, so these readings are taken:
 *   - the rotary table is the caller's: row p = [cos th_0 .. cos th_31, sin th_0 .. sin
 *     th_31] (fp32) for position p;
 *   - the pairs rotated by angle th_i are (2i, 2i+1) (interleaved) or (i, i+32) (halves),
 *     the caller's choice;
 *   - a pair (x, y) becomes (x cos - y sin, y cos + x sin), each product and the sum
 *     rounded to fp32 (no fused multiply-add): the precision in which the kernel decides
 *     the fp8 codes;
 *   - a value v is stored as the e4m3fn code nearest to fp32(v / scale) (ties to the even
 *     code, saturating at +-448), q with q_scale, the cache entry with kv_scale, so that
 *     the decode's dequantisation (code * scale) gives v back;
 *   - slot_mapping[t] = page * page_size + slot names the cache slot of token t's entry;
 *     a negative value means "no entry" (a padding token); a slot outside the cache is an
 *     error and is not written.  A position outside the rotary table is an error: that
 *     token's rope columns (of q and of its entry) are not written.
 * Built with -ffp-contract=off: every float operation below rounds on its own.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

double mlao_fp8_e4m3fn(unsigned code);   /* mla_oracle.c: the format's decode table */

/* bf16 bit pattern -> its exact float value (the high half of a float32 word). */
static float bf16_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* e4m3fn code of the finite value nearest to x; ties go to the even code (even mantissa),
 * which is round-to-nearest-even; beyond +-448 the nearest finite value is +-448 itself,
 * so the search saturates.  NaN -> 0x7F.  The sign of x (of zero too) is kept. */
unsigned mlao_e4m3_encode(double x) {
    if (x != x) return 0x7Fu;
    unsigned sign = signbit(x) ? 0x80u : 0u;
    double a = fabs(x);
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < 0x7Fu; ++c) {   /* 0x00 .. 0x7E: every non-negative finite value */
        double d = fabs(a - mlao_fp8_e4m3fn(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;
}

/* Stored code of value v with per-tensor scale s: the nearest e4m3 of fp32(v / s). */
static uint8_t quantise(float v, float s) {
    float r = v / s;
    return (uint8_t)mlao_e4m3_encode((double)r);
}

/* Rotate the 64 rope values src (bf16 bits) by the table row (cos[32], sin[32]) and write
 * their codes to dst[0..63]. */
static void rope_row(const uint16_t* src, const float* cs, int neox, float scale, uint8_t* dst) {
    for (int i = 0; i < 32; ++i) {
        int a = neox ? i : 2 * i;          /* first and second element of pair i */
        int b = neox ? i + 32 : 2 * i + 1;
        float x = bf16_value(src[a]);
        float y = bf16_value(src[b]);
        float c = cs[i], s = cs[32 + i];
        float xc = x * c, ys = y * s, yc = y * c, xs = x * s;
        float ra = xc - ys;
        float rb = yc + xs;
        dst[a] = quantise(ra, scale);
        dst[b] = quantise(rb, scale);
    }
}

/*
 * q_nope (n_tok, H, 512), q_pe (n_tok, H, 64), kv_c (n_tok, 512), k_pe (n_tok, 64): bf16
 * bits, contiguous.  positions (n_tok,), slot_mapping (n_tok,): int32.  cos_sin
 * (max_pos, 64) fp32.  q_out (n_tok, H, 576) written.  cache: n_slots rows of 576 bytes
 * (slot id = page * page_size + slot, pages contiguous), rows at the mapped slots written.
 * Returns a bit set: 1 = some position outside the table, 2 = some slot outside the cache.
 */
int mlao_rope_concat_cache(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* kv_c,
                           const uint16_t* k_pe, const int32_t* positions, const float* cos_sin,
                           int64_t max_pos, int neox, const int32_t* slot_mapping, float q_scale,
                           float kv_scale, int64_t n_tok, int H, uint8_t* q_out, uint8_t* cache,
                           int64_t n_slots) {
    int err = 0;
    for (int64_t t = 0; t < n_tok; ++t) {
        const int32_t pos = positions[t];
        const int pos_ok = pos >= 0 && (int64_t)pos < max_pos;
        if (!pos_ok) err |= 1;
        const float* cs = pos_ok ? cos_sin + (int64_t)pos * 64 : 0;
        for (int h = 0; h < H; ++h) {
            const int64_t row = t * H + h;
            uint8_t* dst = q_out + row * 576;
            for (int c = 0; c < 512; ++c) dst[c] = quantise(bf16_value(q_nope[row * 512 + c]), q_scale);
            if (pos_ok) rope_row(q_pe + row * 64, cs, neox, q_scale, dst + 512);
        }
        const int32_t slot = slot_mapping[t];
        if (slot < 0) continue;                    /* padding token: no entry */
        if ((int64_t)slot >= n_slots) {
            err |= 2;
            continue;
        }
        uint8_t* dst = cache + (int64_t)slot * 576;
        for (int c = 0; c < 512; ++c) dst[c] = quantise(bf16_value(kv_c[t * 512 + c]), kv_scale);
        if (pos_ok) rope_row(k_pe + t * 64, cs, neox, kv_scale, dst + 512);
    }
    return err;
}
