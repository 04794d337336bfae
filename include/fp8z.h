/*
 * fp8z.h -- C ABI of the block-aware ZeRO-1 optimizer step for blockwise-FP8
 * weights (one GB300, sm_103a).
 *
 * Method (pages cited by title and section):
 *   "A ZeRO Optimizer Design for Blockwise FP8 Quantization" (beipo.top) --
 *     the weight is quantized per 128x128 block ("Blockwise quantization");
 *     main params/grads/moments are folded so every 128x128 block is
 *     contiguous ("Layout transform (fold/unfold)"), then sharded on block
 *     boundaries ("Block-wise split") or by whole params ("Param-wise split");
 *     each DP rank updates its shard element-wise and requantizes the new FP8
 *     weights and scales from its FP32 main params ("Summary").
 *   lpnh.cn "Model-Optimizer" article, §4.3 -- the AdamW update printed as code.
 *   "FP8-Flow-MoE: A Casting-Free FP8 Recipe without Double Quantization
 *     Error", §3.1 -- scale from the block amax and 448, nearest-value rounding,
 *     the E4M3 value formula, power-of-two scales.
 *   mhpn.cn "Core scaling strategies in FP8 training", §3.2 (128x128 block
 *     quantize, scale = 448/amax, clamp to ±448), §4.2 (scale floor 1e-6).
 *
 * Conventions for every call:
 *   - The caller owns all memory.  Device buffers are plain CUDA device
 *     pointers (for instance from PyTorch); host tables are host pointers.  The
 *     library allocates no memory.
 *   - Device calls enqueue work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return at once.  The return value reports argument
 *     and launch errors only.  Errors found on the device (a bad block
 *     descriptor, a wait that ran out of time) are written with an atomic
 *     compare-and-swap into *dev_status (device int32, must start at 0) when
 *     the caller passes one; read it after synchronizing the stream.
 *   - Alignment: float and byte block buffers (p, g, m, v, w_fp8, w_fp8_t,
 *     dequant output) 16 bytes; scale buffers, descriptors and dev_status 4
 *     bytes; the param table 8 bytes.  A misaligned pointer gives FP8Z_EALIGN.
 *   - A block is 128x128 = 16384 elements; float buffers hold
 *     [nblocks,128,128] fp32, row-major inside each block; byte buffers the
 *     same layout of E4M3 codes; scale buffers one fp32 per block.
 *   - Return codes are fp8z_status values; fp8z_status_string() names them.
 *   - The device calls may be captured in a CUDA graph once the same call has
 *     run eagerly on the device (that first call sets the kernels' launch
 *     attributes); scalar arguments such as the hyper-parameters are captured
 *     by value.  fp8z_adamw_requant_step_rowmajor_static is the exception: it
 *     uploads its grad maps from host memory that lives only for the call.
 */
#ifndef FP8Z_H
#define FP8Z_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8Z_API __attribute__((visibility("default")))
#else
#define FP8Z_API
#endif

#define FP8Z_BLOCK 128
#define FP8Z_BLOCK_ELEMS 16384

typedef enum {
    FP8Z_OK = 0,
    FP8Z_EINVAL = -1,        /* bad argument (null, negative, out of range)  */
    FP8Z_EALIGN = -2,        /* pointer not aligned as required              */
    FP8Z_ENOSPACE = -3,      /* a range does not fit the stated capacity     */
    FP8Z_ECUDA = -4,         /* a CUDA runtime call or launch failed         */
    FP8Z_ETIMEOUT = -5,      /* device: a bounded wait ran out of time       */
    FP8Z_EUNSUPPORTED = -6   /* current device is not sm_103 (GB300)         */
} fp8z_status;

typedef enum { FP8Z_SPLIT_BLOCKWISE = 0, FP8Z_SPLIT_PARAMWISE = 1 } fp8z_split;
typedef enum { FP8Z_SCALE_EXACT = 0, FP8Z_SCALE_POW2 = 1 } fp8z_scale_mode;
typedef enum { FP8Z_DECAY_PRE = 0, FP8Z_DECAY_POST = 1 } fp8z_decay_mode;

/* One quantized parameter [e, rows, cols] (e = 1 for a 2-D weight, the expert
 * count for a 3-D expert bank). */
typedef struct { int64_t e, rows, cols; } fp8z_param_shape;

/* Planner output per parameter. */
typedef struct {
    int64_t blk_offset;      /* first folded block of this param in the flat buffer */
    int64_t t_offset;        /* first byte of its column-major [e, cols, rows] copy
                                in a buffer that concatenates all params in order   */
    int64_t t_scale_offset;  /* first entry of its [e, wb, hb] inverse-scale grid    */
    int64_t e, rows, cols;   /* the shape                                            */
    int32_t hb, wb;          /* ceil(rows/128), ceil(cols/128)                        */
    int32_t bucket;          /* DP rank (shard) that owns the param's first block     */
    int32_t reserved;        /* zero                                                  */
} fp8z_param_entry;          /* 64 bytes */

/* One DP shard: blocks [blk_begin, blk_begin + blk_count_real) carry data,
 * [.. + blk_count_real, blk_begin + blk_capacity) are padding. */
typedef struct { int64_t blk_begin, blk_count_real, blk_capacity; } fp8z_shard;

/* One folded block: which param, expert index, block row/col; the valid
 * rows/cols of a ragged edge block (128 inside).  param = -1 and valid = 0
 * for a padding block. */
typedef struct {
    int32_t param, e, brow, bcol;
    uint16_t valid_rows, valid_cols;
} fp8z_block_desc;           /* 20 bytes */

typedef struct {
    int64_t real_elems;              /* sum of e*rows*cols                          */
    int64_t total_blocks;            /* B: folded blocks holding data               */
    int64_t fold_pad_elems;          /* zeros added by padding dims to 128          */
    int64_t shard_pad_elems;         /* (capacity_blocks - B) * 16384               */
    int64_t capacity_blocks;         /* blocks to allocate per state buffer          */
    int64_t naive_straddled_blocks;  /* blocks an even split of the unfolded flat
                                        buffer would cut across ranks                */
} fp8z_plan_summary;

/* AdamW + quantizer hyper-parameters.  The per-step scalars are formed on the
 * host in double from these float values and rounded once to float:
 * step_size = lr/(1-beta1^step), rs_bc2 = 1/sqrt(1-beta2^step),
 * 1-beta1, 1-beta2, decay = 1-lr*weight_decay, lr*weight_decay. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int64_t step;            /* >= 1                                          */
    float fp8_max;           /* (0, 448]; 448 for E4M3                         */
    float min_scale;         /* scale floor, >= 0 (1e-6 in the pages)          */
    int32_t scale_mode;      /* fp8z_scale_mode                                */
    int32_t decay_mode;      /* fp8z_decay_mode                                */
} fp8z_adamw_hparams;        /* 48 bytes */

/*
 * fp8z_plan_shards -- host-only shard planner ("Param-wise split",
 * "Block-wise split" of the ZeRO design page).
 *
 * shapes[nparams] (host) in model order; dp >= 1 shards.
 * BLOCKWISE: every param is padded to multiples of 128 in rows and cols and
 *   folded; params follow each other in the given order, blocks of a param in
 *   (e, block row, block col) order.  With B blocks in all, each shard holds
 *   C = ceil(B/dp) blocks: shard r = [r*C, min((r+1)*C, B)); the tail is padding.
 * PARAMWISE: params sorted by padded block count (descending; ties keep model
 *   order) go one by one to the least-loaded bucket (ties: lowest bucket);
 *   every bucket is padded to the largest load `cap`; bucket r holds blocks
 *   [r*cap, r*cap + load_r), its params in the order they were assigned.
 * Outputs (host, caller-allocated): params_out[nparams], shards_out[dp],
 * summary_out; blocks_out[capacity_blocks] descriptors, or NULL for a size
 * query (summary_out->capacity_blocks tells how many to allocate).
 * Returns FP8Z_OK, FP8Z_EINVAL (bad shape/dp/split/null), FP8Z_ENOSPACE
 * (blocks_cap < capacity_blocks).  Deterministic; no device work.
 */
FP8Z_API int fp8z_plan_shards(const fp8z_param_shape *shapes, int32_t nparams, int32_t dp,
                     int32_t split, fp8z_param_entry *params_out, fp8z_shard *shards_out,
                     fp8z_block_desc *blocks_out, int64_t blocks_cap,
                     fp8z_plan_summary *summary_out);

/*
 * fp8z_adamw_requant_step -- the fused shard step ("Summary" steps: element-wise
 * update of the rank's FP32 main params, then quantize the new FP8 weights and
 * scales from them), for blocks [blk_begin, blk_begin + nblk).
 *
 * Per element, float32, each operation rounded on its own (no FMA):
 *   m' = beta1*m + (1-beta1)*g;  v' = beta2*v + (1-beta2)*(g*g)
 *   u  = m' / (sqrt(v')*rs_bc2 + eps)
 *   PRE : p' = p*decay - step_size*u
 *   POST: p1 = p - step_size*u;  p' = p1 - (lr*wd)*p1
 * Per block: amax = max|p'|; EXACT: s = fp8_max/amax (FLT_MAX if infinite),
 * s = max(s, min_scale), s = 1 when amax == 0; POW2: s = 2^floor(log2(fp8_max/
 * amax)) floored at the smallest power of two >= min_scale; inv = 1/s;
 * q = E4M3(p'*s), round to nearest even, saturated to ±448; NaN stays NaN.
 *
 * p, m, v (updated in place), g: device fp32 [capacity_blocks,128,128].
 * w_fp8: device u8 [capacity_blocks,128,128]; inv_scale: device f32
 *   [capacity_blocks].  Block b of every buffer is the same block.
 * desc: device fp8z_block_desc[capacity_blocks] or NULL.  With desc, element
 *   (r, c) of block b with r >= valid_rows or c >= valid_cols is padding: its
 *   p', m', v' and q are written as 0 and it does not enter the amax.
 * params / nparams: device fp8z_param_entry[nparams] (planner output), needed
 *   only for the column-major copy.
 * w_fp8_t / w_fp8_t_bytes, inv_scale_t / inv_scale_t_count: optional (both
 *   NULL or both set; need desc and params).  For every data block, the
 *   transposed 128x128 tile goes to the param's column-major copy
 *   (w_fp8_t + t_offset + e*cols*rows, element [col][row], ld = rows) and inv
 *   to inv_scale_t[t_scale_offset + e*wb*hb + bcol*hb + brow].  A block whose
 *   destination falls outside the stated sizes is skipped and reported as
 *   FP8Z_EINVAL in *dev_status.
 * hp: host pointer.  dev_status: device int32 or NULL.
 * Returns FP8Z_OK, FP8Z_EINVAL, FP8Z_EALIGN, FP8Z_ENOSPACE (blk_begin+nblk >
 * capacity_blocks), FP8Z_EUNSUPPORTED, FP8Z_ECUDA.  nblk == 0 launches nothing.
 */
FP8Z_API int fp8z_adamw_requant_step(float *p, const float *g, float *m, float *v,
                            uint8_t *w_fp8, float *inv_scale, int64_t capacity_blocks,
                            int64_t blk_begin, int64_t nblk,
                            const fp8z_block_desc *desc,
                            const fp8z_param_entry *params, int32_t nparams,
                            uint8_t *w_fp8_t, int64_t w_fp8_t_bytes,
                            float *inv_scale_t, int64_t inv_scale_t_count,
                            const fp8z_adamw_hparams *hp, int32_t *dev_status,
                            void *stream);

/*
 * fp8z_adamw_requant_step_rowmajor -- the same step with the layout transform
 * fused into it (fold-on-read of the grad, unfold-on-write of the FP8
 * weights).  "A ZeRO Optimizer Design for Blockwise FP8 Quantization",
 * "Summary": the grad is folded before the update and the gathered FP8 params
 * are unfolded after it; "Experiments: performance" names that fold/unfold as
 * the method's extra cost.  Here the kernel reads each block's grad straight
 * from the param's row-major [e, rows, cols] FP32 grad through a TMA tensor
 * map (zero past the ragged edge) and writes the block's E4M3 codes straight
 * into the param's row-major [e, rows, cols] bytes.  p, m, v stay folded (the
 * optimizer's own state), inv_scale is per folded block (already the
 * row-major [e, hb, wb] grid of each param).
 * g_maps: device array of the nparams 128-byte slots (64-byte aligned)
 *   written by fp8z_encode_grad_maps and copied to the device.  Grads whose
 *   cols is not a multiple of 4 are read with plain loads instead of the TMA
 *   engine (slower, same results); a slot that does not match its param entry
 *   gives that param's blocks grad 0 and FP8Z_EINVAL in *dev_status.
 * w_row / w_row_bytes: device buffer of every param's row-major E4M3 bytes,
 *   param i at params[i].t_offset (the same offsets as the column-major copy).
 * desc and params (device) are required.  Other arguments, per-element math,
 * padding and errors as fp8z_adamw_requant_step; a block whose descriptor
 * disagrees with the param table gets grad 0, no row-major write, and
 * FP8Z_EINVAL in *dev_status.
 */
FP8Z_API int fp8z_adamw_requant_step_rowmajor(float *p, float *m, float *v, const void *g_maps,
                                              uint8_t *w_row, int64_t w_row_bytes, float *inv_scale,
                                              int64_t capacity_blocks, int64_t blk_begin, int64_t nblk,
                                              const fp8z_block_desc *desc,
                                              const fp8z_param_entry *params, int32_t nparams,
                                              uint8_t *w_fp8_t, int64_t w_fp8_t_bytes,
                                              float *inv_scale_t, int64_t inv_scale_t_count,
                                              const fp8z_adamw_hparams *hp, int32_t *dev_status,
                                              void *stream);

/*
 * fp8z_adamw_requant_step_rowmajor_static -- fp8z_adamw_requant_step_rowmajor
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a service of the library, not a step of the method.
 *
 * Some callers cannot call cudaMalloc where the step runs: code inside another
 * framework's training step that may only use the tensors that framework hands
 * it, a caller that must not stall the device (an allocation can synchronize
 * it), or one whose device memory is already committed to the optimizer
 * state.  The row-major step needs one piece of working memory besides its
 * inputs and outputs: the grad tensor maps (128 bytes per param) that
 * fp8z_adamw_requant_step_rowmajor reads from a caller-allocated g_maps
 * buffer.  This entry point keeps them instead in an array inside the library
 * (FP8Z_STATIC_GRAD_MAPS maps, 128 KB, held on every device that loads the
 * library until the process exits), so it allocates nothing.
 *
 * g_ptrs: HOST array of nparams device pointers, param i's row-major FP32 grad
 *   [e, rows, cols] (rules as for fp8z_encode_grad_maps).
 * params_host: HOST copy of the planner's param table (the same entries as the
 *   device table `params`); the maps are encoded from it on the host and
 *   copied into the library's array on `stream` before the launch.
 * Every other argument, the arithmetic and the results are exactly those of
 * fp8z_adamw_requant_step_rowmajor.
 * nparams > FP8Z_STATIC_GRAD_MAPS is refused with FP8Z_ENOSPACE, before any
 * device work.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and keeps it.
 * It is not for stream capture (see the conventions above).  Every call shares the one
 * array per device: calls whose work overlaps on the GPU (for instance on two
 * streams) race on it, so issue them in one stream or order them.  The array
 * keeps the maps of the last call.  Calls neither cudaMalloc nor cudaFree nor
 * any routine that allocates device memory.
 */
#define FP8Z_STATIC_GRAD_MAPS 1024
FP8Z_API int fp8z_adamw_requant_step_rowmajor_static(
    float *p, float *m, float *v, const void *const *g_ptrs, const fp8z_param_entry *params_host,
    uint8_t *w_row, int64_t w_row_bytes, float *inv_scale, int64_t capacity_blocks, int64_t blk_begin,
    int64_t nblk, const fp8z_block_desc *desc, const fp8z_param_entry *params, int32_t nparams,
    uint8_t *w_fp8_t, int64_t w_fp8_t_bytes, float *inv_scale_t, int64_t inv_scale_t_count,
    const fp8z_adamw_hparams *hp, int32_t *dev_status, void *stream);

/*
 * fp8z_adamw_requant_step_mx -- the step with an MXFP8 output instead of the
 * 128x128 block scales: E4M3 codes with one E8M0 power-of-two scale per 32
 * consecutive elements of a block row.  "A ZeRO Optimizer Design for Blockwise
 * FP8 Quantization", "Blockwise quantization" (MXFP8 gives memory-contiguous
 * blocks an E8M0 scale); mhpn.cn "Core scaling strategies in FP8 training"
 * §3.1 (32-element blocks share an 8-bit exponent).  Shared exponent
 * x = floor(log2(amax)) - 8, clamped to [-127, 127] (0 for an all-zero
 * group); scale byte = x + 127; code = E4M3(p' / 2^x), nearest even,
 * saturating.  This is the OCP MX rule (the group's largest binade goes to
 * E4M3's largest, [256, 512)): a group whose largest element has a
 * significand above 1.75 maps it into (448, 512) and saturates it to 448,
 * up to ~12.5 % low, where the block-scaled step never saturates.  The
 * block-scaled knobs hp->fp8_max, min_scale and scale_mode do not enter.
 * AdamW, padding, p/g/m/v/w_fp8/desc and errors as
 * fp8z_adamw_requant_step.  mx_scale: device u8 [capacity_blocks, 128, 4]
 * (block b at b*512, row r at r*4), written byte by byte (no alignment
 * needed; nullptr is FP8Z_EINVAL).  Each block needs no block-wide amax, so
 * there is no per-block synchronisation.
 */
FP8Z_API int fp8z_adamw_requant_step_mx(float *p, const float *g, float *m, float *v,
                                        uint8_t *w_fp8, uint8_t *mx_scale, int64_t capacity_blocks,
                                        int64_t blk_begin, int64_t nblk, const fp8z_block_desc *desc,
                                        const fp8z_adamw_hparams *hp, int32_t *dev_status,
                                        void *stream);

/*
 * fp8z_encode_grad_maps -- host only: the 128-byte slots the row-major step
 * reads the grads through.  g_ptrs[i] (host array of device pointers) is
 * param i's row-major FP32 grad [e, rows, cols]; params[i] its planner entry
 * (host).  Writes nparams slots of 128 bytes to maps_out (host, 64-byte
 * aligned); the caller copies them to device memory.  When cols is a multiple
 * of 4 the slot is a TMA tensor map and the grad must be 16-byte aligned;
 * otherwise (a row pitch the TMA engine cannot step over) the slot records
 * the grad's address and shape, the kernel reads that grad with plain loads,
 * and the grad must be 4-byte aligned.  FP8Z_EALIGN for a misaligned grad.
 * The slots must be used with the same param table.  No device work.
 */
FP8Z_API int fp8z_encode_grad_maps(const void *const *g_ptrs, const fp8z_param_entry *params,
                                   int32_t nparams, void *maps_out);

/*
 * fp8z_dequant -- out[b][i] = E4M3_value(w_fp8[b][i]) * inv_scale[b] (float
 * product), for nblk blocks ("FP8-Flow-MoE" §3.1, D(Q(x)) = Q(x)*s).
 * w_fp8: device u8 [nblk,128,128]; inv_scale: device f32 [nblk];
 * out: device f32 [nblk,128,128]; w_fp8 and out 16-byte aligned (they move
 * through the TMA engine as whole blocks).  dev_status: nullable device
 * int32, 4-byte aligned; FP8Z_ETIMEOUT lands there if a bounded wait gave up.
 * Returns FP8Z_OK / EINVAL / EALIGN / ECUDA.
 */
FP8Z_API int fp8z_dequant(const uint8_t *w_fp8, const float *inv_scale, int64_t nblk,
                 float *out, int32_t *dev_status, void *stream);

/*
 * fp8z_transpose_fp8 -- column-major copy of one quantized param.  With
 * 128x128 blocks one scale covers the whole 2-D block, so the layout change is
 * an exact byte permutation and the scale grid is transposed: no dequantize /
 * requantize round trip ("FP8-Flow-MoE" §3.1, scaling-aware transpose).
 * w_fp8 / inv_scale: device, the folded flat buffers; the param's blocks start
 *   at entry->blk_offset.
 * entry: HOST pointer to the param's planner entry (shape, hb, wb, blk_offset).
 * out: device u8 [e, cols, rows] (ld = rows); inv_scale_t: device f32
 *   [e, wb, hb].  out must be 16-byte aligned.  rows a multiple of 16: pairs
 *   of vertically adjacent blocks move through the TMA engine and are written
 *   as 256-byte row pieces (persistent kernel, bounded waits); other row
 *   lengths take a one-CTA-per-block kernel with byte stores at unaligned
 *   edges.
 * dev_status: nullable device int32, 4-byte aligned; FP8Z_ETIMEOUT lands
 *   there if a bounded wait of the TMA kernel gave up.
 * Returns FP8Z_OK / EINVAL / EALIGN / ECUDA.
 */
FP8Z_API int fp8z_transpose_fp8(const uint8_t *w_fp8, const float *inv_scale,
                       const fp8z_param_entry *entry, uint8_t *out, float *inv_scale_t,
                       int32_t *dev_status, void *stream);

/*
 * fp8z_fold / fp8z_unfold -- the layout transform of "A ZeRO Optimizer Design
 * for Blockwise FP8 Quantization", "Layout transform (fold/unfold)": a
 * parameter's row-major [e, rows, cols] tensor <-> its run of contiguous
 * 128x128 blocks in the flat folded buffer (order: expert, block row, block
 * col; row-major inside a block).  Fold writes the padding of ragged edge
 * blocks as zeros ("Block-wise split" pads the quantized dims to multiples of
 * 128); unfold writes only the param's own elements.
 * elem_bytes: 4 (FP32 params, grads, moments) or 1 (E4M3 codes).
 * entry: HOST pointer to the param's planner entry (shape, hb, wb, blk_offset).
 * fold:   src = device [e, rows, cols]; blocks = device base of the folded
 *         buffer (the param's blocks start at entry->blk_offset).
 * unfold: blocks = device base of the folded buffer; dst = device [e, rows, cols].
 * Pointers 16-byte aligned; dev_status as for the step (a wait that gave up).
 * Uses the TMA engine when cols * elem_bytes is a multiple of 16, a plain
 * kernel otherwise.  Returns FP8Z_OK / EINVAL / EALIGN / EUNSUPPORTED / ECUDA.
 * The scale grid needs no unfold: the folded per-block scales are already the
 * row-major [e, hb, wb] grid.
 */
FP8Z_API int fp8z_fold(const void *src, int32_t elem_bytes, const fp8z_param_entry *entry,
                       void *blocks, int32_t *dev_status, void *stream);
FP8Z_API int fp8z_unfold(const void *blocks, int32_t elem_bytes, const fp8z_param_entry *entry,
                         void *dst, int32_t *dev_status, void *stream);

/*
 * fp8z_quantize_rowwise -- 1x128-tile row-wise E4M3 quantization ("FP8-Flow-MoE"
 * §3.1): for each row and each 128 consecutive columns, s = amax/448 (pow2 = 0,
 * kept >= FLT_MIN) or the smallest power of two >= amax/448 (pow2 = 1, kept in
 * [2^-126, 2^127]); s = 1 for a tile of zeros; q = E4M3(x/s), nearest even,
 * saturating.  x: device f32 [rows, cols]; q: device u8 [rows, cols];
 * s: device f32 [rows, cols/128] (dequant multipliers).  cols % 128 == 0.
 * Returns FP8Z_OK / EINVAL / EALIGN / EUNSUPPORTED / ECUDA.
 */
FP8Z_API int fp8z_quantize_rowwise(const float *x, int64_t rows, int64_t cols, int32_t pow2,
                                   uint8_t *q, float *s, void *stream);

/*
 * fp8z_transpose_rowwise -- scaling-aware transpose ("FP8-Flow-MoE" §3.1): the
 * column-wise (1x128 along columns) layout of a row-wise quantized tensor,
 * without dequantizing.  For the 128x128 tile at (row tile i, column tile j)
 * the output scale of each of its 128 output rows is s' = max of the tile's
 * 128 row scales, and q_t[c][r] = E4M3(decode(q[r][c]) * (s[r][j] / s')),
 * computed in FP32 -- with power-of-two scales an exact exponent shift except
 * where the value underflows.  q: device u8 [rows, cols]; s: device f32
 * [rows, cols/128]; q_t: device u8 [cols, rows]; s_t: device f32
 * [cols, rows/128].  rows and cols multiples of 128.
 * Returns FP8Z_OK / EINVAL / EALIGN / EUNSUPPORTED / ECUDA.
 */
FP8Z_API int fp8z_transpose_rowwise(const uint8_t *q, const float *s, int64_t rows, int64_t cols,
                                    uint8_t *q_t, float *s_t, void *stream);

/*
 * fp8z_dequant_rowwise -- row-wise dequantize ("FP8-Flow-MoE" §3.1,
 * D(Q(x)) = Q(x) * s): x[r][c] = E4M3_value(q[r][c]) * s[r][c/128] (float
 * product).  With transpose = 1 the result is written transposed,
 * out[c][r], which is the dequantize-then-transpose half of the naive way to
 * the column-wise layout that the scaling-aware transpose avoids (the other
 * half is fp8z_quantize_rowwise of out).  q: device u8 [rows, cols];
 * s: device f32 [rows, cols/128]; out: device f32 [rows, cols], or
 * [cols, rows] when transposed.  cols a multiple of 128 (rows too when
 * transposed); q and out 16-byte aligned.
 * Returns FP8Z_OK / EINVAL / EALIGN / EUNSUPPORTED / ECUDA.
 */
FP8Z_API int fp8z_dequant_rowwise(const uint8_t *q, const float *s, int64_t rows, int64_t cols,
                                  int32_t transpose, float *out, void *stream);

/*
 * fp8z_e4m3_encode_bits -- out[i] = E4M3 code (round to nearest even,
 * saturating, as in the step) of the float whose bit pattern is
 * first_bits + i, for i < n; n a multiple of 4, out device, 16-byte aligned.
 * Exposes the step's float->E4M3 cast on its own so it can be checked over
 * all 2^32 inputs ("FP8-Flow-MoE" §3.1 value formula).
 */
FP8Z_API int fp8z_e4m3_encode_bits(uint32_t first_bits, int64_t n, uint8_t *out, void *stream);

/*
 * fp8z_watchdog_selftest -- launches one CTA that waits on a barrier nothing
 * will complete, with the same bounded wait the step uses and a limit of
 * timeout_ns nanoseconds; it then writes FP8Z_ETIMEOUT to *dev_status (device
 * int32, starting at 0) and returns.  Lets a test see the device error path
 * without any fault or hang.  timeout_ns in [0, 10^10].
 */
FP8Z_API int fp8z_watchdog_selftest(int32_t *dev_status, int64_t timeout_ns, void *stream);

/*
 * fp8z_set_wait_limit_ns / fp8z_get_wait_limit_ns -- the time limit of every
 * bounded device wait (the barrier waits of the step, dequant, transpose and
 * fold kernels) in launches enqueued after the call.  Process-wide, host only,
 * thread-safe.  ns = 0 restores the default of 2 s; 1 .. 10^10 sets the limit;
 * anything else is FP8Z_EINVAL.  When a wait reaches the limit its kernel
 * writes FP8Z_ETIMEOUT to *dev_status, lets the copies it has in flight land
 * (with a separate limit of 20 s that this setting does not change) and
 * returns; the outputs of that launch are then incomplete.  A very short
 * limit exists to exercise that path in tests and diagnostics; the default
 * is far above any wait of a working launch.
 */
FP8Z_API int fp8z_set_wait_limit_ns(int64_t ns);
FP8Z_API int64_t fp8z_get_wait_limit_ns(void);

/* Static string naming a status code (never NULL). */
FP8Z_API const char *fp8z_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP8Z_H */
