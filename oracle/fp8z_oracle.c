/*
 * fp8z_oracle.c -- plain, slow, single-threaded CPU oracle for the block-aware
 * ZeRO-1 optimizer step on blockwise-FP8 weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The product
 * path (the CUDA library under blockwise_fp8_zero_gb300/) never calls it, and
 * the two share no source, header, table or helper.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (-ffp-contract=off matters: every float product and sum below must round on
 * its own, without being fused into an FMA).
 *
 * Pages followed (cited by title and section throughout):
 *   [ZeRO-BFP8]  "A ZeRO Optimizer Design for Blockwise FP8 Quantization"
 *                (beipo.top/blog/fp8-zero1), sections "Param-wise split",
 *                "Block-wise split", "Layout transform (fold/unfold)", "Summary".
 *   [MO-Quant]   lpnh.cn "Model-Optimizer" article on optimizer-state
 *                quantization, §4.2 (zero-scale guard), §4.3 (AdamW step),
 *                §5.1 (scale==0 pitfall).
 *   [FP8-Flow]   "FP8-Flow-MoE: A Casting-Free FP8 Recipe without Double
 *                Quantization Error", §3.1 (scale = amax/448, round to the
 *                nearest E4M3 value, E4M3 value formula, power-of-two scales).
 *   [FP8-Scale]  mhpn.cn "Core scaling strategies in FP8 training",
 *                §1 (E4M3 range ±448), §3.2 (128x128 block quantize with
 *                scale = 448/amax and a clamp to ±448), §4.2 (scale floor
 *                max(scale, 1e-6)).
 *
 * Readings taken where the pages leave a step open are marked READING.
 *
 * Parity pins (tests/ check this file against things other than itself):
 *   e4m3 encode/decode  -- brute-force nearest search over the decode table
 *                          and torch's float8_e4m3fn cast (library routine).
 *   adamw element step  -- fp64 evaluation of the definition within an error
 *                          bound; closed form at step 1; the torch-op ordering
 *                          printed in [MO-Quant] §4.3 within a few ulp.
 *   scale / quantize    -- amax element maps to exactly ±448; dequant error
 *                          bound; same-layout requant idempotence ([FP8-Flow]
 *                          §3.1); power-of-two layout change is exact.
 *   fold / unfold       -- torch view/permute of [ZeRO-BFP8] "Layout transform".
 *   planner             -- hand-computed tables and invariants.
 *   row-wise 1x128      -- quantizer: brute-force nearest encode of x/s per tile,
 *                          s the smallest power of two >= amax/448 (or amax/448);
 *                          transpose: with power-of-two scales every code moves
 *                          by E' = E - D, M' = M except where it underflows, and
 *                          the double-quantization error of dequantize ->
 *                          transpose -> requantize ([FP8-Flow] §3.1).
 *   MXFP8 step          -- AdamW values equal the block-scaled step's; every
 *                          group's largest element lands in [256, 512) times its
 *                          E8M0 scale; codes equal a brute-force nearest encode
 *                          of p'/2^x; a spike moves only its own group's scale;
 *                          padding and descriptors as in the block-scaled step.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#include <float.h>

#define BLK 128                 /* quantization block edge, [ZeRO-BFP8] "Blockwise quantization" */
#define BLK_ELEMS (BLK * BLK)   /* 16384 elements per folded block */

/* ------------------------------------------------------------------------- */
/* Oracle-side structs.  Field order and widths match the library's ABI so the */
/* same seeded arrays can be handed to both, but nothing here is shared with  */
/* the library's sources.                                                     */
/* ------------------------------------------------------------------------- */
typedef struct { int64_t e, rows, cols; } ref_param_shape;

typedef struct {
    int64_t blk_offset;       /* first folded block of this param            */
    int64_t t_offset;         /* first byte of its column-major copy         */
    int64_t t_scale_offset;   /* first entry of its [E,Wb,Hb] scale grid     */
    int64_t e, rows, cols;    /* shape [E, H=rows, W=cols]                   */
    int32_t hb, wb;           /* blocks along rows / cols                    */
    int32_t bucket;           /* DP shard (bucket) that owns it              */
    int32_t reserved;
} ref_param_entry;

typedef struct { int64_t blk_begin, blk_count_real, blk_capacity; } ref_shard;

typedef struct {
    int32_t param, e, brow, bcol;       /* param = -1 for a padding block    */
    uint16_t valid_rows, valid_cols;
} ref_block_desc;

typedef struct {
    int64_t real_elems, total_blocks, fold_pad_elems, shard_pad_elems,
            capacity_blocks, naive_straddled_blocks;
} ref_plan_summary;

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    float fp8_max, min_scale;
    int32_t scale_mode;   /* 0 = scale = fp8_max/amax, 1 = power of two      */
    int32_t decay_mode;   /* 0 = decay applied to the pre-update param,
                             1 = decay applied after the Adam update          */
} ref_hparams;

/* ------------------------------------------------------------------------- */
/* E4M3 (the "fn" flavour: no infinities, one NaN code per sign, max 448).     */
/* ------------------------------------------------------------------------- */

/* Decode, straight from the value formula of [FP8-Flow] §3.1:
 *   normal  (E>0): (-1)^S * 2^(E-7) * (1 + M/8)
 *   subnormal (E=0): (-1)^S * 2^(-6) * (M/8)        (READING: the page prints
 *   only the normal formula; the subnormal branch is the standard E4M3
 *   definition the page names).  Code 0x7F / 0xFF (E=15, M=7) is NaN, which is
 *   why the largest finite value is 2^8 * 1.75 = 448 ([FP8-Scale] §1). */
double fp8z_ref_e4m3_decode(uint8_t q)
{
    int s = (q >> 7) & 1;
    int E = (q >> 3) & 15;
    int M = q & 7;
    double mag;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        mag = ldexp((double)M / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)M / 8.0, E - 7);
    return s ? -mag : mag;
}

/* Encode one float: round to the nearest E4M3 value, ties to the even
 * mantissa ([FP8-Flow] §3.1 "mapped to the nearest discrete value", RtN),
 * saturating magnitudes above 448 to 448 (the clamp to ±FP8_MAX of
 * [FP8-Scale] §3.2).  NaN -> 0x7F with the input's sign bit; ±Inf -> ±448.
 * Everything is done in double, where every step below is exact. */
uint8_t fp8z_ref_e4m3_encode(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, 4);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)x);
    if (a >= 448.0)                      /* includes +Inf                     */
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;

    /* quantum (spacing of E4M3 values) in the binade that holds a */
    int e2;
    (void)frexp(a, &e2);                 /* a = f * 2^e2, f in [0.5, 1)       */
    int E = e2 - 1;                      /* floor(log2(a))                    */
    double quantum = (E < -6) ? ldexp(1.0, -9) : ldexp(1.0, E - 3);

    double n = a / quantum;              /* exact: power-of-two divisor       */
    double fl = floor(n);
    double frac = n - fl;
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie -> even         */
    double val = r * quantum;            /* nearest E4M3 magnitude            */
    if (val > 448.0)
        val = 448.0;
    if (val == 0.0)
        return sign;

    int code;
    if (val < ldexp(1.0, -6)) {          /* subnormal: val = M * 2^-9         */
        code = (int)(val / ldexp(1.0, -9));
    } else {
        int ev;
        (void)frexp(val, &ev);
        int Ev = ev - 1;                 /* val = (1 + M/8) * 2^Ev            */
        int M = (int)((val / ldexp(1.0, Ev) - 1.0) * 8.0);
        code = ((Ev + 7) << 3) | M;
    }
    return (uint8_t)(sign | code);
}

void fp8z_ref_e4m3_encode_array(const float *x, int64_t n, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = fp8z_ref_e4m3_encode(x[i]);
}

/* Encode the floats whose bit patterns are first, first+1, ..., first+n-1. */
void fp8z_ref_e4m3_encode_bits_range(uint32_t first, int64_t n, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = first + (uint32_t)i;
        float x;
        memcpy(&x, &b, 4);
        q[i] = fp8z_ref_e4m3_encode(x);
    }
}

/* ------------------------------------------------------------------------- */
/* AdamW scalars.                                                              */
/* ------------------------------------------------------------------------- */
/* READING (op order): the hyper-parameters arrive as float32 values.  The
 * per-step scalars are formed in double from those values and rounded to
 * float once, matching the bias-corrected form of [MO-Quant] §4.3:
 *   bc1 = 1 - beta1^t, bc2 = 1 - beta2^t,
 *   step_size = lr / bc1, rs_bc2 = 1 / sqrt(bc2),
 *   omb1 = 1 - beta1, omb2 = 1 - beta2,
 *   decay = 1 - lr*wd, lr_wd = lr*wd.
 * out[] = {beta1, beta2, omb1, omb2, eps, step_size, rs_bc2, decay, lr_wd}. */
void fp8z_ref_adamw_scalars(const ref_hparams *hp, float out[9])
{
    double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
    double t = (double)hp->step;
    double bc1 = 1.0 - pow(b1, t);
    double bc2 = 1.0 - pow(b2, t);
    out[0] = hp->beta1;
    out[1] = hp->beta2;
    out[2] = (float)(1.0 - b1);
    out[3] = (float)(1.0 - b2);
    out[4] = hp->eps;
    out[5] = (float)(lr / bc1);
    out[6] = (float)(1.0 / sqrt(bc2));
    out[7] = (float)(1.0 - lr * wd);
    out[8] = (float)(lr * wd);
}

/* One element of the AdamW update, float32, one rounding per operation.
 * [ZeRO-BFP8] "Summary": the optimizer runs an element-wise update on the
 * rank's FP32 main-param shard; [MO-Quant] §4.3 prints the update:
 *   m' = beta1*m + (1-beta1)*g
 *   v' = beta2*v + (1-beta2)*g*g
 *   d  = sqrt(v') / sqrt(bc2) + eps          (here: sqrt(v') * rs_bc2 + eps)
 *   p' = p - (lr/bc1) * m'/d,   then weight decay.
 * READING (decay position): decay_mode 0 applies it to the pre-update param
 * (p*(1-lr*wd) - step_size*u, the Megatron/torch AdamW form the design builds
 * on); decay_mode 1 applies it after the update, as printed in [MO-Quant]. */
void fp8z_ref_adamw_element(const float sc[9], int decay_mode,
                            float p, float g, float m, float v,
                            float *p_out, float *m_out, float *v_out)
{
    float beta1 = sc[0], beta2 = sc[1], omb1 = sc[2], omb2 = sc[3], eps = sc[4];
    float step_size = sc[5], rs_bc2 = sc[6], decay = sc[7], lr_wd = sc[8];

    float bm = beta1 * m;
    float og = omb1 * g;
    float m1 = bm + og;

    float gg = g * g;
    float bv = beta2 * v;
    float ogg = omb2 * gg;
    float v1 = bv + ogg;

    float sq = sqrtf(v1);
    float sqc = sq * rs_bc2;
    float d = sqc + eps;
    float u = m1 / d;
    float su = step_size * u;

    float p1;
    if (decay_mode == 0) {
        float pd = p * decay;
        p1 = pd - su;
    } else {
        float pu = p - su;
        float dp = lr_wd * pu;
        p1 = pu - dp;
    }
    *p_out = p1;
    *m_out = m1;
    *v_out = v1;
}

/* ------------------------------------------------------------------------- */
/* Per-block scale.                                                            */
/* ------------------------------------------------------------------------- */
/* scale_mode 0: s = fp8_max / amax ([FP8-Scale] §3.2; [FP8-Flow] §3.1 writes
 *   the inverse, amax/448), floored at min_scale ([FP8-Scale] §4.2),
 *   READING: an all-zero block (amax == 0) takes s = 1 ([MO-Quant] §4.2/§5.1
 *   guard), and an infinite quotient (subnormal amax) is clamped to FLT_MAX.
 * scale_mode 1: READING of [FP8-Flow] §3.1 "restrict the scale to a power of
 *   two": s = 2^floor(log2(fp8_max/amax)) taken on the exact quotient, with
 *   the floor rounded up to the next power of two and the top clamped at 2^127.
 * Returns s; *inv = 1/s (IEEE, float). */
float fp8z_ref_block_scale(float amax, float fp8_max, float min_scale,
                           int scale_mode, float *inv)
{
    float s;
    if (amax == 0.0f) {
        s = 1.0f;
    } else if (scale_mode == 0) {
        s = fp8_max / amax;
        if (s > FLT_MAX)
            s = FLT_MAX;
        s = fmaxf(s, min_scale);
    } else {
        /* largest k with 2^k * amax <= fp8_max, searched in double (exact) */
        double a = amax, fm = fp8_max;
        if (isinf(a)) {
            s = 0.0f;
        } else {
            int ea, em;
            double fa = frexp(a, &ea);      /* a = fa * 2^ea                  */
            double ff = frexp(fm, &em);
            int k = em - ea;                /* 2^k*a = fa*2^em vs ff*2^em     */
            if (fa > ff)
                k -= 1;
            if (k > 127)
                k = 127;
            s = (float)ldexp(1.0, k);
        }
        /* floor: smallest power of two >= min_scale */
        int ef;
        double fmn = frexp((double)min_scale, &ef);
        double floor_s = (fmn == 0.5) ? ldexp(1.0, ef - 1) : ldexp(1.0, ef);
        if ((double)s < floor_s)
            s = (float)floor_s;
    }
    *inv = 1.0f / s;
    return s;
}

/* ------------------------------------------------------------------------- */
/* The fused step over a shard's block range.                                  */
/* ------------------------------------------------------------------------- */
/* [ZeRO-BFP8] "Summary": on its shard each DP rank (1) runs the element-wise
 * update on the folded FP32 main params and (2) quantizes the new FP8 params
 * and their scales from the FP32 main params.  Buffers are the flat folded
 * layout [nblk,128,128] (row-major inside a block, [ZeRO-BFP8] "Layout
 * transform").  Block b of every buffer is element range [b*16384, (b+1)*16384),
 * inv_scale[b] its FP32 inverse scale.
 *
 * desc (nullable): per-block descriptor; elements with row >= valid_rows or
 * col >= valid_cols are padding: written as 0 and left out of the amax
 * (READING of the zero padding in "Block-wise split").
 * w_fp8_t / inv_scale_t (nullable, need desc + params): column-major copy of
 * every param in [E, W, H] (ld = H) at params[].t_offset, and its transposed
 * [E, Wb, Hb] inverse-scale grid at params[].t_scale_offset.  For 128x128
 * blocks this is a pure byte permutation ([FP8-Flow] §3.1: one scale per 2-D
 * block is shared by both layouts, so no requantization is needed). */
int fp8z_ref_adamw_requant_step(float *p, const float *g, float *m, float *v,
                                uint8_t *w_fp8, float *inv_scale,
                                int64_t blk_begin, int64_t nblk,
                                const ref_block_desc *desc,
                                const ref_param_entry *params,
                                uint8_t *w_fp8_t, float *inv_scale_t,
                                const ref_hparams *hp)
{
    if (nblk < 0 || blk_begin < 0)
        return -1;
    if ((w_fp8_t || inv_scale_t) && (!desc || !params))
        return -1;
    float sc[9];
    fp8z_ref_adamw_scalars(hp, sc);
    float *pb = (float *)malloc(sizeof(float) * BLK_ELEMS);
    if (!pb)
        return -3;

    for (int64_t b = blk_begin; b < blk_begin + nblk; ++b) {
        int64_t base = b * (int64_t)BLK_ELEMS;
        int vr = BLK, vc = BLK;
        if (desc) {
            vr = desc[b].valid_rows;
            vc = desc[b].valid_cols;
        }
        /* (1) AdamW on every element; padding forced to zero */
        for (int r = 0; r < BLK; ++r) {
            for (int c = 0; c < BLK; ++c) {
                int64_t i = base + r * BLK + c;
                if (r < vr && c < vc) {
                    float p1, m1, v1;
                    fp8z_ref_adamw_element(sc, hp->decay_mode, p[i], g[i], m[i], v[i],
                                           &p1, &m1, &v1);
                    p[i] = p1;
                    m[i] = m1;
                    v[i] = v1;
                    pb[r * BLK + c] = p1;
                } else {
                    p[i] = 0.0f;
                    m[i] = 0.0f;
                    v[i] = 0.0f;
                    pb[r * BLK + c] = 0.0f;
                }
            }
        }
        /* (2) block amax of the updated values ([FP8-Scale] §3.2), valid only */
        float amax = 0.0f;
        for (int r = 0; r < vr; ++r)
            for (int c = 0; c < vc; ++c)
                amax = fmaxf(amax, fabsf(pb[r * BLK + c]));
        float inv;
        float s = fp8z_ref_block_scale(amax, hp->fp8_max, hp->min_scale, hp->scale_mode, &inv);
        /* (3) quantize x*s to E4M3 */
        for (int r = 0; r < BLK; ++r) {
            for (int c = 0; c < BLK; ++c) {
                uint8_t q = 0;
                if (r < vr && c < vc) {
                    float xs = pb[r * BLK + c] * s;
                    q = fp8z_ref_e4m3_encode(xs);
                }
                w_fp8[base + r * BLK + c] = q;
            }
        }
        inv_scale[b] = inv;
        /* (4) optional column-major copy and transposed scale grid */
        if ((w_fp8_t || inv_scale_t) && desc[b].param >= 0) {
            const ref_param_entry *pe = &params[desc[b].param];
            int64_t H = pe->rows, W = pe->cols;
            int64_t e = desc[b].e, br = desc[b].brow, bc = desc[b].bcol;
            if (w_fp8_t) {
                uint8_t *dst = w_fp8_t + pe->t_offset + e * W * H;
                for (int r = 0; r < vr; ++r)
                    for (int c = 0; c < vc; ++c)
                        dst[(bc * BLK + c) * H + br * BLK + r] = w_fp8[base + r * BLK + c];
            }
            if (inv_scale_t)
                inv_scale_t[pe->t_scale_offset + e * (int64_t)pe->wb * pe->hb + bc * pe->hb + br] = inv;
        }
    }
    free(pb);
    return 0;
}

/* Dequantize: x = decode(q) * inv, float product of the exact decoded value
 * and the block's inverse scale ([FP8-Flow] §3.1, D(Q(x)) = Q(x) * s). */
void fp8z_ref_dequant(const uint8_t *w_fp8, const float *inv_scale, int64_t nblk, float *out)
{
    for (int64_t b = 0; b < nblk; ++b)
        for (int64_t i = 0; i < BLK_ELEMS; ++i) {
            int64_t k = b * BLK_ELEMS + i;
            float x = (float)fp8z_ref_e4m3_decode(w_fp8[k]);
            out[k] = x * inv_scale[b];
        }
}

/* Standalone transpose of one param: folded FP8 blocks starting at block
 * pe->blk_offset -> column-major [E, W, H] (ld = H) and the [E, Wb, Hb]
 * inverse-scale grid.  Exact byte permutation (see the step above). */
void fp8z_ref_transpose_fp8(const uint8_t *w_fp8, const float *inv_scale,
                            const ref_param_entry *pe, uint8_t *out, float *inv_scale_t)
{
    int64_t H = pe->rows, W = pe->cols;
    for (int64_t e = 0; e < pe->e; ++e)
        for (int64_t br = 0; br < pe->hb; ++br)
            for (int64_t bc = 0; bc < pe->wb; ++bc) {
                int64_t b = pe->blk_offset + (e * pe->hb + br) * pe->wb + bc;
                for (int r = 0; r < BLK; ++r)
                    for (int c = 0; c < BLK; ++c) {
                        int64_t row = br * BLK + r, col = bc * BLK + c;
                        if (row < H && col < W)
                            out[e * W * H + col * H + row] = w_fp8[b * BLK_ELEMS + r * BLK + c];
                    }
                inv_scale_t[e * pe->wb * pe->hb + bc * pe->hb + br] = inv_scale[b];
            }
}

/* ------------------------------------------------------------------------- */
/* Fold / unfold ([ZeRO-BFP8] "Layout transform (fold/unfold)").               */
/* ------------------------------------------------------------------------- */
/* fold: [E, H, W] row-major -> blocks in (e, hb, wb) order, each block
 * row-major 128x128; rows/cols past H/W are zero ("Block-wise split": the
 * quantized dims are padded to multiples of 128). */
void fp8z_ref_fold(const float *w, int64_t E, int64_t H, int64_t W, float *out)
{
    int64_t Hb = (H + BLK - 1) / BLK, Wb = (W + BLK - 1) / BLK;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t hb = 0; hb < Hb; ++hb)
            for (int64_t wb = 0; wb < Wb; ++wb) {
                int64_t b = (e * Hb + hb) * Wb + wb;
                for (int r = 0; r < BLK; ++r)
                    for (int c = 0; c < BLK; ++c) {
                        int64_t row = hb * BLK + r, col = wb * BLK + c;
                        float x = 0.0f;
                        if (row < H && col < W)
                            x = w[(e * H + row) * W + col];
                        out[b * BLK_ELEMS + r * BLK + c] = x;
                    }
            }
}

/* unfold: inverse of fold, dropping the padding. */
void fp8z_ref_unfold(const float *blocks, int64_t E, int64_t H, int64_t W, float *out)
{
    int64_t Hb = (H + BLK - 1) / BLK, Wb = (W + BLK - 1) / BLK;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t row = 0; row < H; ++row)
            for (int64_t col = 0; col < W; ++col) {
                int64_t b = (e * Hb + row / BLK) * Wb + col / BLK;
                out[(e * H + row) * W + col] =
                    blocks[b * BLK_ELEMS + (row % BLK) * BLK + (col % BLK)];
            }
}

/* ------------------------------------------------------------------------- */
/* Shard planner.                                                              */
/* ------------------------------------------------------------------------- */
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Blocks that an even split of the *unfolded* flat buffer (the plain
 * Megatron/DeepSpeed layout, [ZeRO-BFP8] "Challenges") would cut across two
 * ranks.  Shard size S = ceil(N/dp) elements; a block is cut when any of its
 * 128 row segments crosses a boundary k*S, or when its segments lie in
 * different shards. */
static int64_t naive_straddled(const ref_param_shape *shapes, int32_t n, int32_t dp)
{
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i)
        total += shapes[i].e * shapes[i].rows * shapes[i].cols;
    if (total == 0)
        return 0;
    int64_t S = ceil_div(total, dp);
    int64_t count = 0, off = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t E = shapes[i].e, H = shapes[i].rows, W = shapes[i].cols;
        int64_t Hb = ceil_div(H, BLK), Wb = ceil_div(W, BLK);
        for (int64_t e = 0; e < E; ++e)
            for (int64_t hb = 0; hb < Hb; ++hb)
                for (int64_t wb = 0; wb < Wb; ++wb) {
                    int64_t r0 = hb * BLK, r1 = (hb + 1) * BLK < H ? (hb + 1) * BLK : H;
                    int64_t c0 = wb * BLK, c1 = (wb + 1) * BLK < W ? (wb + 1) * BLK : W;
                    int64_t first = off + (e * H + r0) * W + c0;
                    int64_t last = off + (e * H + r1 - 1) * W + c1 - 1;
                    int64_t shard0 = first / S;
                    int cut = 0;
                    for (int64_t r = r0; r < r1 && !cut; ++r) {
                        int64_t a = off + (e * H + r) * W + c0;
                        int64_t z = off + (e * H + r) * W + c1 - 1;
                        if (a / S != shard0 || z / S != shard0)
                            cut = 1;
                    }
                    (void)last;
                    count += cut;
                }
        off += E * H * W;
    }
    return count;
}

/* Fill param entries, block descriptors and summary.
 * split 0 = block-wise ([ZeRO-BFP8] "Block-wise split"): params in the given
 *   order, each padded to multiples of 128 and folded; the flat block list is
 *   cut into dp shards of C = ceil(B/dp) blocks, the last ones padded.
 * split 1 = param-wise ([ZeRO-BFP8] "Param-wise split"): READING -- params
 *   sorted by padded block count, descending, ties by lower index (stable);
 *   each goes to the bucket with the least load so far, ties to the lowest
 *   bucket; every bucket is padded to the largest load; bucket r occupies
 *   blocks [r*cap, r*cap + load_r) with its params in assignment order.
 * blocks_out == NULL: only params/shards/summary are written (size query).
 * Return 0, or -1 bad args, -3 blocks_cap too small. */
int fp8z_ref_plan_shards(const ref_param_shape *shapes, int32_t nparams, int32_t dp,
                         int32_t split, ref_param_entry *params_out, ref_shard *shards_out,
                         ref_block_desc *blocks_out, int64_t blocks_cap,
                         ref_plan_summary *summary_out)
{
    if (nparams < 0 || dp <= 0 || (split != 0 && split != 1) || !params_out ||
        !shards_out || !summary_out || (nparams > 0 && !shapes))
        return -1;
    for (int32_t i = 0; i < nparams; ++i)
        if (shapes[i].e <= 0 || shapes[i].rows <= 0 || shapes[i].cols <= 0)
            return -1;

    int64_t real = 0, fold_pad = 0, B = 0, t_off = 0, ts_off = 0;
    int64_t *nb = (int64_t *)calloc((size_t)(nparams > 0 ? nparams : 1), sizeof(int64_t));
    if (!nb)
        return -3;
    for (int32_t i = 0; i < nparams; ++i) {
        int64_t E = shapes[i].e, H = shapes[i].rows, W = shapes[i].cols;
        int64_t Hb = ceil_div(H, BLK), Wb = ceil_div(W, BLK);
        ref_param_entry *pe = &params_out[i];
        memset(pe, 0, sizeof(*pe));
        pe->e = E; pe->rows = H; pe->cols = W;
        pe->hb = (int32_t)Hb; pe->wb = (int32_t)Wb;
        pe->t_offset = t_off;
        pe->t_scale_offset = ts_off;
        nb[i] = E * Hb * Wb;
        real += E * H * W;
        fold_pad += E * Hb * BLK * Wb * BLK - E * H * W;
        B += nb[i];
        t_off += E * H * W;
        ts_off += E * Hb * Wb;
    }

    int64_t cap;
    if (split == 0) {
        cap = ceil_div(B, dp);
        int64_t off = 0;
        for (int32_t i = 0; i < nparams; ++i) {
            params_out[i].blk_offset = off;
            params_out[i].bucket = cap > 0 ? (int32_t)(off / cap) : 0;
            off += nb[i];
        }
        for (int32_t r = 0; r < dp; ++r) {
            int64_t b0 = (int64_t)r * cap;
            int64_t cnt = B - b0;
            if (cnt < 0) cnt = 0;
            if (cnt > cap) cnt = cap;
            shards_out[r].blk_begin = b0;
            shards_out[r].blk_count_real = cnt;
            shards_out[r].blk_capacity = cap;
        }
    } else {
        int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nparams > 0 ? nparams : 1));
        int64_t *load = (int64_t *)calloc((size_t)dp, sizeof(int64_t));
        if (!order || !load) {
            free(order); free(load); free(nb);
            return -3;
        }
        for (int32_t i = 0; i < nparams; ++i)
            order[i] = i;
        /* stable insertion sort, descending padded block count */
        for (int32_t i = 1; i < nparams; ++i) {
            int32_t x = order[i];
            int32_t j = i - 1;
            while (j >= 0 && nb[order[j]] < nb[x]) {
                order[j + 1] = order[j];
                --j;
            }
            order[j + 1] = x;
        }
        for (int32_t k = 0; k < nparams; ++k) {
            int32_t i = order[k];
            int32_t best = 0;
            for (int32_t r = 1; r < dp; ++r)
                if (load[r] < load[best])
                    best = r;
            params_out[i].bucket = best;
            params_out[i].blk_offset = load[best];   /* relative for now */
            load[best] += nb[i];
        }
        cap = 0;
        for (int32_t r = 0; r < dp; ++r)
            if (load[r] > cap)
                cap = load[r];
        for (int32_t i = 0; i < nparams; ++i)
            params_out[i].blk_offset += (int64_t)params_out[i].bucket * cap;
        for (int32_t r = 0; r < dp; ++r) {
            shards_out[r].blk_begin = (int64_t)r * cap;
            shards_out[r].blk_count_real = load[r];
            shards_out[r].blk_capacity = cap;
        }
        free(order);
        free(load);
    }

    int64_t capacity = (int64_t)dp * cap;
    summary_out->real_elems = real;
    summary_out->total_blocks = B;
    summary_out->fold_pad_elems = fold_pad;
    summary_out->shard_pad_elems = (capacity - B) * BLK_ELEMS;
    summary_out->capacity_blocks = capacity;
    summary_out->naive_straddled_blocks = naive_straddled(shapes, nparams, dp);

    if (blocks_out) {
        if (blocks_cap < capacity) {
            free(nb);
            return -3;
        }
        for (int64_t b = 0; b < capacity; ++b) {
            blocks_out[b].param = -1;
            blocks_out[b].e = 0;
            blocks_out[b].brow = 0;
            blocks_out[b].bcol = 0;
            blocks_out[b].valid_rows = 0;
            blocks_out[b].valid_cols = 0;
        }
        for (int32_t i = 0; i < nparams; ++i) {
            const ref_param_entry *pe = &params_out[i];
            for (int64_t e = 0; e < pe->e; ++e)
                for (int64_t hb = 0; hb < pe->hb; ++hb)
                    for (int64_t wb = 0; wb < pe->wb; ++wb) {
                        int64_t b = pe->blk_offset + (e * pe->hb + hb) * pe->wb + wb;
                        int64_t vr = pe->rows - hb * BLK, vc = pe->cols - wb * BLK;
                        blocks_out[b].param = i;
                        blocks_out[b].e = (int32_t)e;
                        blocks_out[b].brow = (int32_t)hb;
                        blocks_out[b].bcol = (int32_t)wb;
                        blocks_out[b].valid_rows = (uint16_t)(vr > BLK ? BLK : vr);
                        blocks_out[b].valid_cols = (uint16_t)(vc > BLK ? BLK : vc);
                    }
        }
    }
    free(nb);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* 1x128-tile row-wise quantization and the scaling-aware transpose.           */
/* ------------------------------------------------------------------------- */
/* [FP8-Flow] §3.1: a row-wise quantized tensor has one scale per 128
 * consecutive elements of a row, s = amax/448 (the dequant multiplier), and
 * Q(x) = round(x/s) to the nearest E4M3 value.  With power-of-two scales
 * (s = 2^T) re-expressing a value under another power-of-two scale only moves
 * its exponent.  READING: pow2 = 1 takes s = 2^ceil(log2(amax/448)), the
 * smallest power of two that keeps every |x/s| <= 448; a tile of zeros takes
 * s = 1; scales stay within the normal float range.
 * q: [R, C] codes, s: [R, C/128] scales, C a multiple of 128. */
void fp8z_ref_quantize_rowwise(const float *x, int64_t R, int64_t C, int pow2,
                               uint8_t *q, float *s)
{
    int64_t nt = C / BLK;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t t = 0; t < nt; ++t) {
            const float *xr = x + r * C + t * BLK;
            float amax = 0.0f;
            for (int c = 0; c < BLK; ++c)
                amax = fmaxf(amax, fabsf(xr[c]));
            double sc;
            if (amax == 0.0f) {
                sc = 1.0;
            } else if (pow2) {
                /* smallest 2^k >= amax/448, on the exact quotient, kept within
                 * the normal float range [2^-126, 2^127] */
                double ratio = (double)amax / 448.0;
                int k = 127;                          /* an infinite amax takes the clamp (READING) */
                if (!isinf(ratio)) {
                    int e;
                    double f = frexp(ratio, &e);      /* ratio = f * 2^e, f in [0.5,1) */
                    k = (f == 0.5) ? e - 1 : e;
                }
                if (k < -126) k = -126;
                if (k > 127) k = 127;
                sc = ldexp(1.0, k);
            } else {
                /* amax/448 in float, kept at least the smallest normal float */
                sc = (double)fmaxf(amax / 448.0f, FLT_MIN);
            }
            s[r * nt + t] = (float)sc;
            for (int c = 0; c < BLK; ++c)
                q[r * C + t * BLK + c] = fp8z_ref_e4m3_encode((float)((double)xr[c] / (double)(float)sc));
        }
}

/* Scaling-aware transpose ([FP8-Flow] §3.1): the column-wise layout of the same
 * tensor, without going back to high precision.  For the 128x128 tile at
 * (row tile i, column tile j), every output row c (an input column) takes the
 * scale s' = max over the tile's 128 input rows of s[r][j] (aligning to the
 * largest scale avoids overflow), and each code is re-expressed under it:
 * q'[c][r] = nearest E4M3 value to decode(q[r][c]) * s[r][j] / s'.  With
 * power-of-two scales this is the page's exponent shift E' = E - D, M' = M
 * (D = log2 s' - log2 s[r][j]), exact unless the shifted value leaves the
 * normal range; then it rounds to the nearest subnormal (ties to even).
 * READING: the re-expression is computed in FP32 -- ratio = s[r][j] / s',
 * y = decode(q) * ratio, one rounding of y to E4M3 -- every step of which is
 * exact for power-of-two scales.
 * q_t: [C, R] codes, s_t: [C, R/128] scales; R and C multiples of 128. */
void fp8z_ref_transpose_rowwise(const uint8_t *q, const float *s, int64_t R, int64_t C,
                                uint8_t *q_t, float *s_t)
{
    int64_t ntc = C / BLK, ntr = R / BLK;
    for (int64_t i = 0; i < ntr; ++i)
        for (int64_t j = 0; j < ntc; ++j) {
            float smax = 0.0f;
            for (int r = 0; r < BLK; ++r)
                smax = fmaxf(smax, s[(i * BLK + r) * ntc + j]);
            for (int c = 0; c < BLK; ++c) {
                int64_t oc = j * BLK + c;
                s_t[oc * ntr + i] = smax;
                for (int r = 0; r < BLK; ++r) {
                    int64_t ir = i * BLK + r;
                    float v = (float)fp8z_ref_e4m3_decode(q[ir * C + oc]);
                    float ratio = s[ir * ntc + j] / smax;
                    float y = v * ratio;
                    q_t[oc * R + ir] = fp8z_ref_e4m3_encode(y);
                }
            }
        }
}

/* Row-wise dequantize: x[r][c] = decode(q[r][c]) * s[r][c/128] (float). */
void fp8z_ref_dequant_rowwise(const uint8_t *q, const float *s, int64_t R, int64_t C, float *x)
{
    int64_t nt = C / BLK;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            x[r * C + c] = (float)fp8z_ref_e4m3_decode(q[r * C + c]) * s[r * nt + c / BLK];
}

/* ------------------------------------------------------------------------- */
/* MXFP8 output: E4M3 codes with one E8M0 power-of-two scale per 32 elements.  */
/* ------------------------------------------------------------------------- */
/* [ZeRO-BFP8] "Blockwise quantization": MXFP8 gives each memory-contiguous
 * block an E8M0 scale; [FP8-Scale] §3.1: 32-element blocks share an 8-bit
 * exponent, value = element * 2^(exponent - bias).  READING: the shared
 * exponent of a group of 32 consecutive elements of a block row is
 * floor(log2(amax)) - 8 (8 = the largest E4M3 exponent, 448 = 1.75 * 2^8),
 * clamped to [-127, 127]; E8M0 code = exponent + 127; an all-zero group takes
 * exponent 0.  Elements are E4M3(x / 2^exponent), nearest even, saturating at
 * ±448 (the largest element lands in [256, 512)).  Padding (desc) is zero and
 * enters the amax as zero.
 * mx_scale: [nblk, 128, 4] bytes (block b at b*512, row r at r*4). */
int fp8z_ref_adamw_requant_step_mx(float *p, const float *g, float *m, float *v,
                                   uint8_t *w_fp8, uint8_t *mx_scale,
                                   int64_t blk_begin, int64_t nblk,
                                   const ref_block_desc *desc, const ref_hparams *hp)
{
    if (nblk < 0 || blk_begin < 0)
        return -1;
    float sc[9];
    fp8z_ref_adamw_scalars(hp, sc);
    for (int64_t b = blk_begin; b < blk_begin + nblk; ++b) {
        int64_t base = b * (int64_t)BLK_ELEMS;
        int vr = BLK, vc = BLK;
        if (desc) {
            vr = desc[b].valid_rows;
            vc = desc[b].valid_cols;
        }
        for (int r = 0; r < BLK; ++r) {
            float row[BLK];
            for (int c = 0; c < BLK; ++c) {
                int64_t i = base + r * BLK + c;
                if (r < vr && c < vc) {
                    float p1, m1, v1;
                    fp8z_ref_adamw_element(sc, hp->decay_mode, p[i], g[i], m[i], v[i], &p1, &m1, &v1);
                    p[i] = p1; m[i] = m1; v[i] = v1;
                    row[c] = p1;
                } else {
                    p[i] = 0.0f; m[i] = 0.0f; v[i] = 0.0f;
                    row[c] = 0.0f;
                }
            }
            for (int gi = 0; gi < BLK / 32; ++gi) {
                float amax = 0.0f;
                for (int c = 0; c < 32; ++c)
                    amax = fmaxf(amax, fabsf(row[gi * 32 + c]));
                int ex = 0;
                if (isinf(amax)) {
                    ex = 127;                           /* floor(log2(+Inf)) - 8, clamped (READING) */
                } else if (amax > 0.0f) {
                    int e2;
                    (void)frexp((double)amax, &e2);     /* amax = f * 2^e2, f in [0.5,1) */
                    ex = (e2 - 1) - 8;
                    if (ex < -127) ex = -127;
                    if (ex > 127) ex = 127;
                }
                mx_scale[b * 512 + r * 4 + gi] = (uint8_t)(ex + 127);
                for (int c = 0; c < 32; ++c) {
                    int cc = gi * 32 + c;
                    float y = (float)((double)row[cc] / ldexp(1.0, ex));
                    w_fp8[base + r * BLK + cc] = (r < vr && cc < vc) ? fp8z_ref_e4m3_encode(y) : 0;
                }
            }
        }
    }
    return 0;
}
