// fold.cu -- fold / unfold between a parameter's row-major [E, H, W] layout
// and the flat buffer of contiguous 128x128 blocks (sm_103a).
//
// "A ZeRO Optimizer Design for Blockwise FP8 Quantization", "Layout transform
// (fold/unfold)": fold turns the row-major weight into 128x128 blocks laid out
// one after another (order e, block row, block col), so the ZeRO-1 optimizer can
// split it on block boundaries; unfold is the inverse, applied to the gathered
// FP8 weights after the step.  The quantized dims are zero-padded to multiples
// of 128 ("Block-wise split").
//
// GB300 design: both directions are pure data movement (HBM-bound, 2 x element
// size per element).  A folded block is one contiguous 16384-element run and in
// the row-major tensor a 128x128 tile, so each CTA moves whole blocks with the
// TMA engine: fold = one tiled tensor-map load of the tile (the engine fills the
// ragged edge with zeros) + one bulk store of the contiguous block; unfold =
// one bulk load + one tiled tensor-map store (the engine clips at the tensor's
// edge).  Persistent CTAs keep rings of blocks in flight (FP32: one CTA per
// SM, 192 KB; bytes: two CTAs per SM, 80 KB each, one store in flight beside
// the loads); the byte unfold moves two blocks per store (256-byte row
// pieces).  Shapes
// whose row pitch is not a multiple of 16 bytes (a TMA rule) take a plain
// kernel instead.
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fp8z.h"
#include "fp8z_device.cuh"
#include "fp8z_host.h"

namespace fp8z {
namespace {

constexpr int kBlk = FP8Z_BLOCK;
constexpr int kBlkElems = FP8Z_BLOCK_ELEMS;

struct FoldArgs {
    uint8_t* flat;            // first block of the param in the folded buffer
    int64_t hb, wb, nblk;     // blocks per row / col of one expert matrix, total
    int32_t esz;              // element size in bytes (1 or 4)
    int32_t nbuf;             // ring buffers of one block each
    int32_t* dev_status;
    int64_t timeout_ns;
};

// Block b of the param -> (x, y, z) of its tile in the row-major tensor.
__device__ __forceinline__ void tile_coords(const FoldArgs& F, int64_t b, int& x, int& y, int& z) {
    const int64_t per = F.hb * F.wb;
    z = int(b / per);
    const int64_t r = b % per;
    y = int((r / F.wb) * kBlk);
    x = int((r % F.wb) * kBlk);
}

// One thread per CTA drives the copies.  Blocks are dealt round-robin over a
// persistent grid; each CTA keeps a ring of nbuf block buffers: kLag of them
// may still be read by their stores while nbuf - 1 - kLag hold loads in flight
// and one is being written out.  FP32 blocks (64 KB): one CTA per SM with a
// 192 KB ring (3 buffers, no store slack); byte blocks (16 KB): two CTAs per
// SM with 80 KB rings, three loads ahead and one store in flight.  Measured on
// GB300, fractions of the copy bandwidth, E4M3 unfold / fold: at 32 x 7168^2
// 0.963 / 0.959 against 0.946 / 0.947 for three CTAs with 64 KB rings and no
// slack (two loads ahead 0.940, four 0.945; one CTA with a 192 KB ring
// 0.925); at 117 x 7168^2 every one of these runs the unfold at 0.941 and the
// fold at 0.945-0.950.
constexpr int kRingBytesF32 = 192 * 1024;
constexpr int kStoreLagF32 = 0;
constexpr int kRingBytesU8 = 80 * 1024;
constexpr int kCtasPerSmU8 = 2;
constexpr int kStoreLagU8 = 1;

template <bool kFold, int kLag>
__global__ void __launch_bounds__(32) fold_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                      const FoldArgs F) {
    extern __shared__ __align__(1024) unsigned char smem[];
    if (threadIdx.x != 0) return;
    const uint32_t box = uint32_t(kBlkElems) * F.esz;
    const int nbuf = F.nbuf;                              // 3 (fp32) or 5 (bytes)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(nbuf) * box);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + nbuf);
    const uint32_t buf0 = smem_addr(smem);
    const uint32_t bar0 = smem_addr(bars);
    *abort_flag = 0;
    for (int i = 0; i < nbuf; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
    const Watchdog wd{abort_flag, F.dev_status, F.timeout_ns};

    const int64_t count = (F.nblk - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= nblk
    auto blk = [&](int64_t i) { return int64_t(blockIdx.x) + i * gridDim.x; };
    auto issue_load = [&](int64_t i) {
        const int s = int(i % nbuf);
        const uint32_t dst = buf0 + s * box;
        mbar_arrive_expect_tx(bar0 + 8 * s, box);
        if (kFold) {
            int x, y, z;
            tile_coords(F, blk(i), x, y, z);
            tma_load_3d(dst, &map, x, y, z, bar0 + 8 * s);
        } else {
            bulk_g2s_nohint(dst, F.flat + blk(i) * int64_t(box), box, bar0 + 8 * s);
        }
    };

    const int64_t ahead = nbuf - 1 - kLag;                // >= 1 (host checks)
    for (int64_t i = 0; i < count && i < ahead; ++i) issue_load(i);
    for (int64_t i = 0; i < count; ++i) {
        const int64_t j = i + ahead;
        if (j < count) {
            // block j reuses the buffer of block i-1-kLag: at most the kLag
            // newest store groups (blocks i-kLag..i-1) may still be reading
            bulk_wait_read<kLag>();
            issue_load(j);
        }
        const int s = int(i % nbuf);
        if (!mbar_wait_bounded(bar0 + 8 * s, uint32_t((i / nbuf) & 1), wd)) {
            // let every load still in flight land before the CTA leaves:
            // block i (the one that timed out) up to the newest issued, j
            for (int64_t k = i; k < count && k <= j; ++k)
                mbar_wait_drain(bar0 + 8 * int(k % nbuf), uint32_t((k / nbuf) & 1), F.dev_status);
            bulk_wait_all();
            return;
        }
        fence_proxy_async();
        const uint32_t src = buf0 + s * box;
        if (kFold) {
            bulk_s2g(F.flat + blk(i) * int64_t(box), src, box);
        } else {
            int x, y, z;
            tile_coords(F, blk(i), x, y, z);
            tma_store_3d(&map, x, y, z, src);
        }
        bulk_commit();
    }
    bulk_wait_all();
}

// Byte unfold of block pairs.  One tensor-map load brings two horizontally
// adjacent blocks with their rows interleaved ([row][block][128 bytes]; the
// map is a permuted view of the folded buffer: x, then block at a 16 KB
// stride, then row at a 128-byte stride), and one 256-byte-wide tensor-map
// store writes them, so every output row piece is 256 contiguous bytes
// instead of 128.  An odd last block column loads the next block (or the zero
// fill past the param) beside it, and the store clips it at the tensor's edge.
// Two CTAs per SM, rings of three 32 KB pairs, one store in flight beside one
// load ahead.  Measured on GB300 at 117 x 7168^2: 1.855 ms against 1.912 ms
// for the one-block kernel above (0.972 against 0.943 of the copy bandwidth;
// one CTA with six pairs ran no faster than the one-block kernel, two CTAs
// with no store slack 1.880 ms, three CTAs with two pairs 1.865 ms).
constexpr int kPairBytes = 2 * kBlkElems;
constexpr int kPairRing = 3 * kPairBytes;
constexpr int kPairCtasPerSm = 2;
constexpr int kPairLag = 1;
static_assert(kPairRing / kPairBytes - 1 - kPairLag >= 1, "pair ring too small");

struct PairArgs {
    int64_t hb, wb, wp, nitems;   // block rows / cols of one expert, pairs per block row, pairs in all
    int32_t* dev_status;
    int64_t timeout_ns;
};

__global__ void __launch_bounds__(32) unfold_pair_kernel(const __grid_constant__ CUtensorMap in_map,
                                                         const __grid_constant__ CUtensorMap out_map,
                                                         const PairArgs P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    if (threadIdx.x != 0) return;
    constexpr int nbuf = kPairRing / kPairBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + nbuf);
    const uint32_t buf0 = smem_addr(smem);
    const uint32_t bar0 = smem_addr(bars);
    *abort_flag = 0;
    for (int i = 0; i < nbuf; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
    const Watchdog wd{abort_flag, P.dev_status, P.timeout_ns};

    const int64_t count = (P.nitems - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= nitems
    // pair i of this CTA -> expert, block row, pair index within the block row
    auto coords = [&](int64_t i, int64_t& e, int64_t& brow, int64_t& pr) {
        const int64_t it = int64_t(blockIdx.x) + i * gridDim.x;
        const int64_t per = P.hb * P.wp;
        e = it / per;
        brow = (it % per) / P.wp;
        pr = it % P.wp;
    };
    auto issue_load = [&](int64_t i) {
        const int s = int(i % nbuf);
        int64_t e, brow, pr;
        coords(i, e, brow, pr);
        mbar_arrive_expect_tx(bar0 + 8 * s, kPairBytes);
        tma_load_3d(buf0 + s * kPairBytes, &in_map, 0, int((e * P.hb + brow) * P.wb + 2 * pr), 0, bar0 + 8 * s);
    };

    const int64_t ahead = nbuf - 1 - kPairLag;
    for (int64_t i = 0; i < count && i < ahead; ++i) issue_load(i);
    for (int64_t i = 0; i < count; ++i) {
        const int64_t j = i + ahead;
        if (j < count) {
            // pair j reuses the buffer of pair i-1-kLag: at most the kLag
            // newest store groups (pairs i-kLag..i-1) may still be reading
            bulk_wait_read<kPairLag>();
            issue_load(j);
        }
        const int s = int(i % nbuf);
        if (!mbar_wait_bounded(bar0 + 8 * s, uint32_t((i / nbuf) & 1), wd)) {
            // let every load still in flight land before the CTA leaves:
            // pair i (the one that timed out) up to the newest issued, j
            for (int64_t k = i; k < count && k <= j; ++k)
                mbar_wait_drain(bar0 + 8 * int(k % nbuf), uint32_t((k / nbuf) & 1), P.dev_status);
            bulk_wait_all();
            return;
        }
        fence_proxy_async();
        int64_t e, brow, pr;
        coords(i, e, brow, pr);
        tma_store_3d(&out_map, int(2 * pr * kBlk), int(brow * kBlk), int(e), buf0 + s * kPairBytes);
        bulk_commit();
    }
    bulk_wait_all();
}

// Plain path for shapes the TMA engine cannot address (row pitch not a
// multiple of 16 bytes): one CTA per block, rows of the tile read/written by
// consecutive threads.
template <bool kFold, typename T>
__global__ void __launch_bounds__(256) fold_plain_kernel(const T* __restrict__ src, T* __restrict__ dst,
                                                         int64_t H, int64_t W, int64_t hb, int64_t wb) {
    const int64_t b = blockIdx.x;
    const int64_t per = hb * wb;
    const int64_t e = b / per, r = b % per;
    const int64_t row0 = (r / wb) * kBlk, col0 = (r % wb) * kBlk;
    const T* in = kFold ? src : src + b * kBlkElems;
    T* out = kFold ? dst + b * kBlkElems : dst;
    for (int i = threadIdx.x; i < kBlkElems; i += blockDim.x) {
        const int rr = i / kBlk, cc = i % kBlk;
        const int64_t row = row0 + rr, col = col0 + cc;
        const bool inside = row < H && col < W;
        const int64_t g = (e * H + row) * W + col;
        if (kFold) {
            out[i] = inside ? in[g] : T(0);
        } else if (inside) {
            out[g] = in[i];
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(host::tensor_map_encoder());
}

int run(bool fold, const void* src, int32_t esz, const fp8z_param_entry* entry, void* dst,
        int32_t* dev_status, void* stream) {
    if (!src || !dst || !entry || (esz != 1 && esz != 4)) return FP8Z_EINVAL;
    const fp8z_param_entry& pe = *entry;
    if (pe.e < 1 || pe.rows < 1 || pe.cols < 1 || pe.blk_offset < 0) return FP8Z_EINVAL;
    if (pe.hb != (pe.rows + kBlk - 1) / kBlk || pe.wb != (pe.cols + kBlk - 1) / kBlk) return FP8Z_EINVAL;
    const int64_t nblk = pe.e * pe.hb * pe.wb;
    if (nblk > 0x7FFFFFFFLL || pe.e > 0x7FFFFFFFLL) return FP8Z_EINVAL;
    if (!host::aligned(src, 16) || !host::aligned(dst, 16) || !host::aligned(dev_status, 4))
        return FP8Z_EALIGN;
    int sms = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* flat_c = static_cast<const uint8_t*>(fold ? dst : src) + pe.blk_offset * int64_t(kBlkElems) * esz;
    uint8_t* flat = const_cast<uint8_t*>(flat_c);
    void* rowmajor = const_cast<void*>(fold ? src : dst);

    const bool tma_ok = (pe.cols * esz) % 16 == 0 && pe.rows <= 0xFFFFFFFFLL && pe.cols <= 0xFFFFFFFFLL;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tma_ok ? encode_fn() : nullptr;
    if (enc && !fold && esz == 1) {
        // byte unfold by block pairs (falls through to the one-block kernel if
        // the driver refuses either map)
        CUtensorMap in_map, out_map;
        std::memset(&in_map, 0, sizeof(in_map));
        std::memset(&out_map, 0, sizeof(out_map));
        const cuuint64_t in_dims[3] = {cuuint64_t(kBlk), cuuint64_t(nblk), cuuint64_t(kBlk)};
        const cuuint64_t in_strides[2] = {cuuint64_t(kBlkElems), cuuint64_t(kBlk)};
        const cuuint32_t in_box[3] = {kBlk, 2, kBlk};
        const cuuint64_t out_dims[3] = {cuuint64_t(pe.cols), cuuint64_t(pe.rows), cuuint64_t(pe.e)};
        const cuuint64_t out_strides[2] = {cuuint64_t(pe.cols), cuuint64_t(pe.rows * pe.cols)};
        const cuuint32_t out_box[3] = {2 * kBlk, kBlk, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&in_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, flat, in_dims, in_strides, in_box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
            enc(&out_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, rowmajor, out_dims, out_strides, out_box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            const int smem = kPairRing + (kPairRing / kPairBytes) * 8 + 16;
            rc = host::set_smem_once(reinterpret_cast<const void*>(&unfold_pair_kernel), 9, smem);
            if (rc != FP8Z_OK) return rc;
            const int64_t wp = (pe.wb + 1) / 2;
            const PairArgs P{pe.hb, pe.wb, wp, pe.e * pe.hb * wp, dev_status, host::wait_limit_ns()};
            const int64_t cap = int64_t(sms) * kPairCtasPerSm;
            const unsigned grid = unsigned(P.nitems < cap ? P.nitems : cap);
            unfold_pair_kernel<<<grid, 32, smem, st>>>(in_map, out_map, P);
            return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
        }
    }
    if (enc) {
        CUtensorMap map;
        std::memset(&map, 0, sizeof(map));
        const cuuint64_t dims[3] = {cuuint64_t(pe.cols), cuuint64_t(pe.rows), cuuint64_t(pe.e)};
        const cuuint64_t strides[2] = {cuuint64_t(pe.cols * esz), cuuint64_t(pe.rows * pe.cols * esz)};
        const cuuint32_t boxd[3] = {kBlk, kBlk, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        const CUresult cr = enc(&map, esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                3, rowmajor, dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr == CUDA_SUCCESS) {
            const bool f32 = esz == 4;
            const int ring = f32 ? kRingBytesF32 : kRingBytesU8;
            const int nbuf = ring / (kBlkElems * esz);
            static_assert(kRingBytesF32 / (kBlkElems * 4) - 1 - kStoreLagF32 >= 1, "FP32 ring too small");
            static_assert(kRingBytesU8 / kBlkElems - 1 - kStoreLagU8 >= 1, "byte ring too small");
            FoldArgs F{flat, pe.hb, pe.wb, nblk, esz, nbuf, dev_status, host::wait_limit_ns()};
            const int smem = ring + nbuf * 8 + 16;
            const void* k = fold ? (f32 ? reinterpret_cast<const void*>(&fold_tma_kernel<true, kStoreLagF32>)
                                        : reinterpret_cast<const void*>(&fold_tma_kernel<true, kStoreLagU8>))
                                 : (f32 ? reinterpret_cast<const void*>(&fold_tma_kernel<false, kStoreLagF32>)
                                        : reinterpret_cast<const void*>(&fold_tma_kernel<false, kStoreLagU8>));
            rc = host::set_smem_once(k, fold ? (f32 ? 2 : 7) : (f32 ? 3 : 8), smem);
            if (rc != FP8Z_OK) return rc;
            const int64_t cap = int64_t(sms) * (f32 ? 1 : kCtasPerSmU8);
            const unsigned grid = unsigned(nblk < cap ? nblk : cap);
            if (fold && f32)
                fold_tma_kernel<true, kStoreLagF32><<<grid, 32, smem, st>>>(map, F);
            else if (fold)
                fold_tma_kernel<true, kStoreLagU8><<<grid, 32, smem, st>>>(map, F);
            else if (f32)
                fold_tma_kernel<false, kStoreLagF32><<<grid, 32, smem, st>>>(map, F);
            else
                fold_tma_kernel<false, kStoreLagU8><<<grid, 32, smem, st>>>(map, F);
            return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
        }
    }
    // plain path
    const unsigned grid = unsigned(nblk);
    if (esz == 4) {
        if (fold)
            fold_plain_kernel<true, float><<<grid, 256, 0, st>>>(static_cast<const float*>(src),
                                                                 reinterpret_cast<float*>(flat), pe.rows,
                                                                 pe.cols, pe.hb, pe.wb);
        else
            fold_plain_kernel<false, float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(flat),
                                                                  static_cast<float*>(dst), pe.rows, pe.cols,
                                                                  pe.hb, pe.wb);
    } else {
        if (fold)
            fold_plain_kernel<true, uint8_t><<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(src), flat,
                                                                   pe.rows, pe.cols, pe.hb, pe.wb);
        else
            fold_plain_kernel<false, uint8_t><<<grid, 256, 0, st>>>(flat, static_cast<uint8_t*>(dst),
                                                                    pe.rows, pe.cols, pe.hb, pe.wb);
    }
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

}  // namespace
}  // namespace fp8z

extern "C" int fp8z_fold(const void* src, int32_t elem_bytes, const fp8z_param_entry* entry,
                         void* blocks, int32_t* dev_status, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_fold");
    return fp8z::run(true, src, elem_bytes, entry, blocks, dev_status, stream);
}

extern "C" int fp8z_unfold(const void* blocks, int32_t elem_bytes, const fp8z_param_entry* entry,
                           void* dst, int32_t* dev_status, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_unfold");
    return fp8z::run(false, blocks, elem_bytes, entry, dst, dev_status, stream);
}
