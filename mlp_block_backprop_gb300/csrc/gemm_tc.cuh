// gemm_tc.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with the
// block's fused prologue/epilogues.
//
//   D[M,N] = sum_k A[m,k] * B[n,k]      bf16 operands, fp32 accumulator in TMEM
//
// A and B are each either K-major (stored [rows][K]) or MN-major (stored [K][rows]);
// the tensor core reads both layouts straight from shared memory, so the
// transposed products of the backward pass (g.B and A^T.g of the MatMul rule of
// "Reverse-mode automatic differentiation", section 5) need no transpose copies.
//
// CTA layout (persistent over output tiles):
//   warp 0      TMA producer: A/B tiles -> shared-memory ring of kStages stages
//   warp 1      owns TMEM; one lane issues tcgen05.mma (K = 16 per instruction)
//   warps 2..5  epilogue: TMEM -> registers -> fused math -> shared -> TMA store
//               (warps 2..9 for the residual, gate and fp32-output epilogues: two
//               warps per TMEM lane quarter, each taking half of a tile's columns)
//   warps 6..9  (the in-GEMM RMSNorm variant of the forward W1 GEMM only) sum of
//               x^2 per row, read from each A stage once its MMAs have completed
//               (then the stage goes back to the producer), gives rstd for the
//               epilogue; works with pair tiles, each CTA summing its own rows
//   warps 6..9  (the wgrad-W1 GEMM with side rows only) RMSNorm backward rows,
//               independent of the tensor-core pipeline (side_norm_rows)
// The accumulator is double buffered in TMEM (2 x BN columns) so the epilogue of
// one tile overlaps the main loop of the next.
//
// Work is a list of segments per worker (a CTA, or a CTA pair): whole tiles dealt
// round robin, then optionally a contiguous range of the remaining tiles' k-blocks
// ("stream-K", see SegIter), so every worker ends at the same time.  A tile split
// between workers is finished by the one holding its first k-blocks from the
// others' fp32 partial sums; the fp32 += epilogues simply add every segment.
//
// Two tile modes:
//   single (PAIR = false): one CTA per SM computes a 128 x BN tile.
//   pair   (PAIR = true):  a cluster of two CTAs on two SMs computes a 256 x BN
//     tile with tcgen05.mma.cta_group::2.  Each CTA loads its 128 rows of A and
//     BN/2 rows of B; the leader CTA (rank 0) issues the MMAs, which read both
//     CTAs' shared memory; each CTA's TMEM receives its own 128 rows.  Per SM this
//     stages half of B per unit of tensor work, which is what keeps the tensor
//     core fed when the stage refill rate, not the MMA, is the limit.
#pragma once

#include "ptx.cuh"

namespace mlpblk {

constexpr int kBM = 128;      // rows per CTA (UMMA M per CTA)
constexpr int kSmemLimit = 232448;  // 227 KB dynamic shared memory per CTA
// Accumulator buffers of a pair tile (256 TMEM columns each): two, so the
// epilogue of one tile overlaps the main loop of the next.
constexpr int kPairAccBufs = 2;

template <int BN_, int EPI_, bool A_MN_, bool B_MN_, bool PAIR_ = false, bool F8_ = false>
struct GemmCfg {
    static constexpr int BN = BN_;               // tile width (of the pair tile in pair mode)
    static constexpr int EPI = EPI_;
    static constexpr bool A_MN = A_MN_;
    static constexpr bool B_MN = B_MN_;
    static constexpr bool PAIR = PAIR_;
    // operand element type: bf16 (kind::f16) or E4M3 (kind::f8f6f4).  A stage row
    // is 128 bytes either way: 64 bf16 or 128 E4M3 values of K, and one MMA
    // takes 32 bytes of K per row (16 or 32 values)
    static constexpr bool F8 = F8_;
    static constexpr int kElem = F8 ? 1 : 2;
    static constexpr int kBKe = 128 / kElem;       // K values per stage
    static constexpr int kUmmaKe = 32 / kElem;     // K values per tcgen05.mma
    static constexpr int kMNBox = 128 / kElem;     // MN values per MN-major box row
    static constexpr int kMNBoxBytes = kBKe * 128; // one MN-major box: kBKe rows of 128 bytes
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;  // rows of one output tile
    static constexpr int kBRows = PAIR ? BN / 2 : BN;    // rows of B staged per CTA
    static constexpr bool kNorm = (EPI == kEpiFwdW1);
    static constexpr bool kReluSq = (EPI == kEpiFwdW1 || EPI == kEpiFwdW1Pre || EPI == kEpiFwdW1A);
    static constexpr bool kAOnly = (EPI == kEpiFwdW1A);  // a out only (h is not kept)
    static constexpr bool kOutBf16 = (kReluSq || EPI == kEpiFwdW2 || EPI == kEpiDgradH || EPI == kEpiStoreBf16);
    static constexpr bool kSide = (EPI == kEpiAccF32ColScaleNorm);  // + RMSNorm backward side warps
    static constexpr bool kColScale = (EPI == kEpiAccF32ColScale || kSide);
    static constexpr bool kReduce = (EPI == kEpiAccF32 || kColScale);
    static constexpr int kNumOut = (kReluSq && !kAOnly) ? 2 : 1;
    static constexpr int kChunkCols = kOutBf16 ? 64 : 32;  // 128 bytes of a row per chunk
    static constexpr int kNumChunks = BN / kChunkCols;
    // epilogue warps: one per TMEM lane quarter, or two (each draining half of a
    // tile's columns) for the epilogues that also read an [M][N] bf16 operand, whose
    // per-element work is the largest, and for the fp32 outputs, whose last tile's
    // 128 KB per CTA ends the kernel (the 120M-class block's dgrad-n 38.3 -> 36.8
    // us); the two-output W1 epilogue measured no faster so
    static constexpr bool kF32x8 = (EPI == kEpiStoreF32 || EPI == kEpiAccF32 || EPI == kEpiAccF32ColScale);
    static constexpr int kEpiWarps = (EPI == kEpiFwdW2 || EPI == kEpiDgradH || kF32x8) ? 8 : 4;
    static constexpr int kThreads = kNorm ? 320 : 64 + 32 * kEpiWarps + (kSide ? 32 * kSideWarps : 0);
    static constexpr int kABytes = kBM * 128;
    static constexpr int kBBytes = kBRows * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    // epilogues that read a [M][N] bf16 operand (x for the residual, h for the
    // gate) prefetch each warp's 32 rows of the next tile into shared memory and
    // stage their output in place of it, so they need no staging buffers
    static constexpr bool kAux = (EPI == kEpiFwdW2 || EPI == kEpiDgradH);
    static constexpr int kAuxBytes = kAux ? 4 * kNumChunks * 4096 : 0;
    // output staging per epilogue warp and output: double buffered, except for
    // the two-output W1 epilogue and the eight-warp fp32 epilogues, whose shared
    // memory goes to a deeper pipeline
    static constexpr int kStagingBufs = (kNumOut == 2 || kF32x8) ? 1 : 2;
    static constexpr int kStagingBytes = kAux ? 0 : kEpiWarps * kNumOut * kStagingBufs * 4096;
    // per-row scale read from args.rstd_in (1 when that is null)
    static constexpr bool kRowScale = (EPI == kEpiDgradH || EPI == kEpiFwdW1Pre || EPI == kEpiFwdW1A ||
                                       EPI == kEpiStoreF32 || EPI == kEpiStoreBf16);
    static constexpr int kCtrlBytes = 1024 + (kNorm ? 1024 : 0);  // barriers (+ rstd[2][128])
    static constexpr int kAlignSlack = 1024;
    static constexpr int kStagesRaw =
        (kSmemLimit - kAlignSlack - kCtrlBytes - kStagingBytes - kAuxBytes) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kSmemBytes =
        kAlignSlack + kCtrlBytes + kStagingBytes + kAuxBytes + kStages * kStageBytes;
    // TMEM accumulator buffers (pair tiles: see kPairAccBufs)
    static constexpr int kAccBufs = PAIR ? kPairAccBufs : 2;
    // TMEM columns allocated: a power of two >= the accumulators' columns
    static constexpr uint32_t kTmemCols = kAccBufs * BN <= 256 ? 256u : 512u;
    static constexpr uint32_t kIdesc = F8 ? idesc_e4m3_f32(kTileM, BN, A_MN, B_MN)
                                          : idesc_bf16_f32(kTileM, BN, A_MN, B_MN);
    static_assert(kStages >= 2, "not enough shared memory for a pipeline");
    // a split tile's owner copies one partial sum (128 x BN fp32) into the
    // pipeline stages, which its last segment has finished with
    static_assert(kStages * kStageBytes >= 4 * BN * 128, "stages cannot hold a partial tile");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory over budget");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
    // a pair stages BN/2 rows of B per CTA; MN-major B is staged in 64-wide
    // swizzle blocks, so there BN/2 must be a multiple of 64
    static_assert(!PAIR || BN == 256 || (BN == 192 && !B_MN), "pair tiles are 256 x 256 or 256 x 192");
    static_assert(!B_MN || kBRows % kMNBox == 0, "MN-major B is staged in whole 128-byte box rows");
};

// One segment of a worker's work: k-blocks [kb0, kb1) of one output tile.
struct Seg {
    int tile, m0, n0, n_blk, kb0, kb1;  // m0, n0: origin of the (pair) output tile
    int crow;  // K-grouped: rows added to the output row (the expert's block of C)
    int boff;  // M-grouped: the expert's offset into B (rows of a K-major B, K of an MN-major B)
};

// First stream-K iteration of worker w (iterations of the tiles after dp_tiles,
// k-block fastest).
__device__ __forceinline__ int sk_begin(const GemmArgs &a, int w) {
    return min(w * a.sk_base + min(w, a.sk_rem), a.sk_total);
}

// A worker's segments in order: its whole tiles w, w + workers, ... below
// dp_tiles, then its stream-K range, cut at tile boundaries.  Only the first
// stream-K segment can start inside a tile, and only the last can end inside
// one, so a worker writes at most one partial and owns at most one split tile.
//
// Grouped GEMMs (the routed experts; whole tiles only):
//   M-grouped: the rows are the experts' token segments back to back, each padded
//     to a multiple of 256 rows (grp_rows[e] .. grp_rows[e+1]); the row count is
//     read from device memory, and a tile's expert selects its slice of B;
//   K-grouped (weight gradients): expert e's tiles sum over K = its segment's
//     rows and write the expert's block of C; experts without tokens are skipped.
struct SegIter {
    int worker, j, n_dp, pos, end, m_tiles;
    int dp_tiles, sk_base, sk_rem, sk_total;  // the schedule (device-computed when M-grouped and split)
    int sub_j, sub_n;                         // k-parts of the last tiles (GemmArgs::sub_parts)
};

__device__ __forceinline__ int sk_begin(const SegIter &it, int w) {
    return min(w * it.sk_base + min(w, it.sk_rem), it.sk_total);
}

template <int TILE_M>
__device__ __forceinline__ SegIter seg_begin(const GemmArgs &a, int worker) {
    SegIter it;
    it.worker = worker;
    it.j = 0;
    it.m_tiles = a.m_tiles;
    it.dp_tiles = a.dp_tiles;
    it.sk_base = a.sk_base;
    it.sk_rem = a.sk_rem;
    it.sk_total = a.sk_total;
    it.sub_j = it.sub_n = 0;
    if (a.grp_mode == kGroupM && a.grp_split) {
        // M-grouped with the split schedule: the host's rule (whole-tile rounds
        // while more than two remain, then the k-blocks split evenly) applied to
        // the tile count the routing left in device memory
        it.m_tiles = a.grp_rows[a.grp_count] / TILE_M;
        const int tiles = it.m_tiles * a.n_tiles;
        const int full = tiles / a.workers;
        if (tiles % a.workers == 0) {
            it.dp_tiles = tiles;
        } else {
            it.dp_tiles = full >= 2 ? (full - 1) * a.workers : 0;
        }
        it.sk_total = (tiles - it.dp_tiles) * a.k_blocks;
        it.sk_base = it.sk_total / a.workers;
        it.sk_rem = it.sk_total % a.workers;
        it.n_dp = it.dp_tiles / a.workers;
        it.pos = sk_begin(it, worker);
        it.end = sk_begin(it, worker + 1);
        return it;
    }
    if (a.grp_mode != kGroupNone) {
        if (a.grp_mode == kGroupM) it.m_tiles = a.grp_rows[a.grp_count] / TILE_M;
        const int total = (a.grp_mode == kGroupM ? it.m_tiles : a.grp_count * a.m_tiles) * a.n_tiles;
        it.n_dp = total > worker ? (total - worker + a.workers - 1) / a.workers : 0;
        it.pos = it.end = 0;
        return it;
    }
    it.n_dp = a.dp_tiles / a.workers;
    if (a.sub_parts > 0) {
        const int items = (a.tiles - a.dp_tiles) * a.sub_parts;
        it.sub_n = items > worker ? (items - worker + a.workers - 1) / a.workers : 0;
        it.pos = it.end = 0;
        return it;
    }
    it.pos = sk_begin(a, worker);
    it.end = sk_begin(a, worker + 1);
    return it;
}

// Tiles are rastered in groups of group_m M-tiles that sweep all N-tiles
// together, so tiles in flight at the same time share operand tiles in L2.
template <int BN, int TILE_M, int KBE>
__device__ __forceinline__ bool seg_next(const GemmArgs &a, SegIter &it, Seg &s) {
    while (true) {
        int t;
        if (it.j < it.n_dp) {
            t = it.worker + it.j * a.workers;
            s.kb0 = 0;
            s.kb1 = a.k_blocks;
            ++it.j;
        } else if (it.sub_j < it.sub_n) {
            // k-part `part` of tile dp_tiles + i: the parts go round robin, part by part
            const int item = it.worker + it.sub_j * a.workers;
            const int rem = a.tiles - it.dp_tiles;
            const int part = item / rem;
            t = it.dp_tiles + (item - part * rem);
            s.kb0 = part * a.sub_kb;
            s.kb1 = min(a.k_blocks, s.kb0 + a.sub_kb);
            ++it.sub_j;
        } else if (it.pos < it.end) {
            const int tt = it.pos / a.k_blocks;
            s.kb0 = it.pos - tt * a.k_blocks;
            s.kb1 = min(a.k_blocks, s.kb0 + (it.end - it.pos));
            it.pos += s.kb1 - s.kb0;
            t = it.dp_tiles + tt;
        } else {
            return false;
        }
        s.tile = t;
        s.crow = 0;
        s.boff = 0;
        if (a.grp_mode == kGroupK) {
            const int per = a.m_tiles * a.n_tiles;
            const int e = t / per;
            t -= e * per;
            s.kb0 = a.grp_rows[e] / KBE;
            s.kb1 = a.grp_rows[e + 1] / KBE;
            if (s.kb0 == s.kb1) continue;  // an expert without tokens: no tile
            s.crow = e * a.grp_c_off;
        }
        int mi = 0, ni = 0;
        raster_tile(t, it.m_tiles, a.n_tiles, a.group_m, mi, ni);
        s.n_blk = ni;
        s.m0 = mi * TILE_M;
        s.n0 = ni * BN;
        if (a.grp_mode == kGroupM) {
            int e = 0;
            while (e + 1 < a.grp_count && a.grp_rows[e + 1] <= s.m0) ++e;
            s.boff = e * a.grp_b_off;
        }
        return true;
    }
}

__device__ __forceinline__ float sq(float v) { return v * v; }

// Sum of squares of the 8 bf16 values in a 16-byte vector.
__device__ __forceinline__ float sumsq_bf16x8(uint4 v) {
    return sq(bf16_lo(v.x)) + sq(bf16_hi(v.x)) + sq(bf16_lo(v.y)) + sq(bf16_hi(v.y)) +
           sq(bf16_lo(v.z)) + sq(bf16_hi(v.z)) + sq(bf16_lo(v.w)) + sq(bf16_hi(v.w));
}

// RMSNorm backward with the residual gradient for the rows of the side warps
// (warp sw of kSideWarps in each CTA; rows sw + kSideWarps*blockIdx.x + k*stride),
// on dn_s = rstd*dn:  dx = dy + gamma*dn_s - x*c,  c = r^2 * mean_k(gamma*dn_s*x),
// dgamma partial += dn_s*x.  One row per warp at a time: lane l owns the 8-column
// chunks l, l+32, l+64 (d <= kSideNormMaxD), the row sum is a shuffle butterfly.
// The CTA's side warps then add their dgamma shares into the CTA's partial row
// in warp order (a fixed order, as in the row kernel).  Once every CTA's row is
// complete (an arrival count), warp 0 of CTA b adds the partial rows of the
// 8-column chunks b, b + grid, ... into dgamma: lane l sums rows l, l + 32, ...
// and a butterfly over the lanes finishes, so the order is fixed by the grid.
// The GEMM's warps do not wait for any of this.
__device__ __forceinline__ void side_norm_rows(const SideNorm &sn, int sw, volatile int *abort) {
    constexpr int kCPT = kSideNormMaxD / 256;
    const int lane = threadIdx.x & 31;
    const int d = sn.d;
    const int chunks = d / 8;
    griddep_wait();  // dn_s: written by the previous kernel
    uint4 g[kCPT];
    float acc[kCPT][8];
#pragma unroll
    for (int j = 0; j < kCPT; ++j) {
        const int q = lane + 32 * j;
        g[j] = q < chunks ? ld_global_nc_v4(sn.gamma + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
    }
    const float inv_d = 1.0f / static_cast<float>(d);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kSideWarps;
    // the loop is bound by load latency (one row in flight per warp): lane 0
    // asks L2 for the rows kAhead strides ahead, so the row loads hit L2
    constexpr int kAhead = 2;
    const uint32_t row_bytes = static_cast<uint32_t>(d) * 2;
    const int64_t t_first = static_cast<int64_t>(blockIdx.x) * kSideWarps + sw;
    if (lane == 0)
        for (int ahead = 0; ahead < kAhead; ++ahead) {
            const int64_t tp = t_first + ahead * stride;
            if (tp < sn.T) {
                bulk_prefetch_l2(sn.x + tp * d, row_bytes);
                bulk_prefetch_l2(sn.dy + tp * d, row_bytes);
                bulk_prefetch_l2(sn.dn_s + tp * d, row_bytes);
            }
        }
    for (int64_t t = t_first; t < sn.T; t += stride) {
        if (lane == 0 && t + kAhead * stride < sn.T) {
            const int64_t tp = t + kAhead * stride;
            bulk_prefetch_l2(sn.x + tp * d, row_bytes);
            bulk_prefetch_l2(sn.dy + tp * d, row_bytes);
            bulk_prefetch_l2(sn.dn_s + tp * d, row_bytes);
        }
        const float r = sn.rstd[t];
        uint4 xv[kCPT], yv[kCPT];
        float nv[kCPT][8];
#pragma unroll
        for (int j = 0; j < kCPT; ++j) {
            const int q = lane + 32 * j;
            if (q < chunks) {
                const int64_t off = t * d + 8 * q;
                xv[j] = ld_global_nc_v4(sn.x + off);
                yv[j] = ld_global_nc_v4(sn.dy + off);
                const uint4 n0 = ld_global_nc_v4(sn.dn_s + off);  // 8 bf16 values
                nv[j][0] = bf16_lo(n0.x); nv[j][1] = bf16_hi(n0.x);
                nv[j][2] = bf16_lo(n0.y); nv[j][3] = bf16_hi(n0.y);
                nv[j][4] = bf16_lo(n0.z); nv[j][5] = bf16_hi(n0.z);
                nv[j][6] = bf16_lo(n0.w); nv[j][7] = bf16_hi(n0.w);
            } else {
                xv[j] = yv[j] = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int i = 0; i < 8; ++i) nv[j][i] = 0.0f;
            }
        }
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < kCPT; ++j) {
            const uint32_t gw[4] = {g[j].x, g[j].y, g[j].z, g[j].w};
            const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                s += bf16_lo(gw[i]) * nv[j][2 * i] * bf16_lo(xw[i]) + bf16_hi(gw[i]) * nv[j][2 * i + 1] * bf16_hi(xw[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float cr = r * r * s * inv_d;
#pragma unroll
        for (int j = 0; j < kCPT; ++j) {
            const int q = lane + 32 * j;
            if (q >= chunks) continue;
            const uint32_t gw[4] = {g[j].x, g[j].y, g[j].z, g[j].w};
            const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
            const uint32_t yw[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x0 = bf16_lo(xw[i]), x1 = bf16_hi(xw[i]);
                const float n0 = nv[j][2 * i], n1 = nv[j][2 * i + 1];
                o[i] = pack_bf16x2(bf16_lo(yw[i]) + bf16_lo(gw[i]) * n0 - x0 * cr,
                                   bf16_hi(yw[i]) + bf16_hi(gw[i]) * n1 - x1 * cr);
                acc[j][2 * i] += n0 * x0;
                acc[j][2 * i + 1] += n1 * x1;
            }
            st_global_v4(sn.dx + t * d + 8 * q, o[0], o[1], o[2], o[3]);
        }
    }
    // the CTA's dgamma partial row: side warp 0 stores its share, then each
    // next warp adds its own, in warp order
    float *out = sn.part + static_cast<int64_t>(blockIdx.x) * d;
    for (int w = 0; w < kSideWarps; ++w) {
        named_barrier_sync(1, 32 * kSideWarps);
        if (w == sw) {
#pragma unroll
            for (int j = 0; j < kCPT; ++j) {
                const int q = lane + 32 * j;
                if (q >= chunks) continue;
                float *p = out + 8 * q;
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = acc[j][i];
                if (w > 0) {
                    const float4 a0 = ld_global_cg_v4(p), a1 = ld_global_cg_v4(p + 4);
                    v[0] += a0.x; v[1] += a0.y; v[2] += a0.z; v[3] += a0.w;
                    v[4] += a1.x; v[5] += a1.y; v[6] += a1.z; v[7] += a1.w;
                }
                st_global_v4(p, v[0], v[1], v[2], v[3]);
                st_global_v4(p + 4, v[4], v[5], v[6], v[7]);
            }
            __threadfence_block();
        }
    }
    // the row is complete (the barrier orders every side warp's stores before
    // the release of the one arrival; a reader's acquire of the count sees them)
    named_barrier_sync(1, 32 * kSideWarps);
    if (sw != 0) return;
    if (lane == 0) red_release_gpu_add(sn.arrive, 1);
    const int P = static_cast<int>(gridDim.x);
    if (static_cast<int>(blockIdx.x) >= chunks) return;
    // this CTA's first chunk of dgamma, read before the wait (nothing else writes it)
    float g0[8];
    if (lane == 0) {
        const float *dg = sn.dgamma + 8 * blockIdx.x;
#pragma unroll
        for (int i = 0; i < 8; ++i) g0[i] = dg[i];
    }
    // one lane polls (with a pause between polls), then every lane acquires
    int ok = 1;
    if (lane == 0) ok = count_wait_sleep(sn.arrive, P, abort);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    (void)ld_acquire_gpu(sn.arrive);
    constexpr int kRowsPerLane = (kMaxSkSlots + 31) / 32;
    for (int q = blockIdx.x; q < chunks; q += P) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        // every lane's rows in flight at once (one pass while P <= kMaxSkSlots)
        for (int p0 = 0; p0 < P; p0 += 32 * kRowsPerLane) {
            float4 a[kRowsPerLane][2];
#pragma unroll
            for (int k = 0; k < kRowsPerLane; ++k) {
                const int p = p0 + lane + 32 * k;
                if (p < P) {
                    const float *src = sn.part + static_cast<int64_t>(p) * d + 8 * q;
                    a[k][0] = ld_global_cg_v4(src);
                    a[k][1] = ld_global_cg_v4(src + 4);
                } else {
                    a[k][0] = a[k][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
            }
#pragma unroll
            for (int k = 0; k < kRowsPerLane; ++k) {
                v[0] += a[k][0].x; v[1] += a[k][0].y; v[2] += a[k][0].z; v[3] += a[k][0].w;
                v[4] += a[k][1].x; v[5] += a[k][1].y; v[6] += a[k][1].z; v[7] += a[k][1].w;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
        if (lane == 0) {
            float *dg = sn.dgamma + 8 * q;
            if (q == static_cast<int>(blockIdx.x)) {
#pragma unroll
                for (int i = 0; i < 8; ++i) dg[i] = g0[i] + v[i];
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) dg[i] += v[i];
            }
        }
    }
}

// What the roles of a CTA share: its shared-memory carve-up and identities.
struct CtaCtx {
    uint8_t *stages, *staging, *aux_smem;
    uint64_t *full_bar, *empty_bar, *accf_bar, *acce_bar, *aux_bar, *consumed_bar;
    volatile int *abort_flag;
    float *rs;
    uint32_t tmem_base, rank;
    bool leader;
    int worker, slot, warp, lane;
};

// TMA producer (one thread): the segments' A and B k-blocks into the ring of S
// stages; `stage` and `phase` carry the ring position from call to call.
template <class C, int S>
__device__ __forceinline__ void producer_run(const CUtensorMap *pA, const CUtensorMap *pB, const GemmArgs &args,
                                             const CtaCtx &x, int &stage, uint32_t &phase) {
    uint8_t *stages = x.stages, *staging = x.staging, *aux_smem = x.aux_smem;
    uint64_t *full_bar = x.full_bar, *empty_bar = x.empty_bar, *accf_bar = x.accf_bar, *acce_bar = x.acce_bar,
             *aux_bar = x.aux_bar, *consumed_bar = x.consumed_bar;
    volatile int *abort_flag = x.abort_flag;
    float *rs = x.rs;
    const uint32_t tmem_base = x.tmem_base, rank = x.rank;
    const bool leader = x.leader;
    const int worker = x.worker, slot = x.slot, warp = x.warp, lane = x.lane;
    (void)stages; (void)staging; (void)aux_smem; (void)full_bar; (void)empty_bar; (void)accf_bar;
    (void)acce_bar; (void)aux_bar; (void)consumed_bar; (void)abort_flag; (void)rs; (void)tmem_base;
    (void)rank; (void)leader; (void)worker; (void)slot; (void)warp; (void)lane;
    SegIter si = seg_begin<C::kTileM>(args, worker);
    Seg w;
    while (seg_next<C::BN, C::kTileM, C::kBKe>(args, si, w)) {
        const int a_row = w.m0 + static_cast<int>(rank) * kBM;       // this CTA's A rows
        // this CTA's B rows (a K-major B's rows carry the expert offset)
        const int b_row = w.n0 + static_cast<int>(rank) * C::kBRows + (C::B_MN ? 0 : w.boff);
        const int bk = C::B_MN ? w.boff : 0;  // an MN-major B's K carries it
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) return;
            uint8_t *sa = stages + stage * C::kStageBytes;
            uint8_t *sb = sa + C::kABytes;
            const int k0 = kb * C::kBKe;
            // where this CTA's A and B loads signal completion
            uint32_t bar_a = smem_u32(&full_bar[stage]), bar_b = bar_a;
            bool a_pair = false, b_pair = false;
            if (!C::PAIR) {
                mbar_arrive_expect_tx(&full_bar[stage], C::kStageBytes);
            } else if (leader) {
                // the leader's barrier collects both CTAs' bytes
                mbar_arrive_expect_tx(&full_bar[stage], 2 * C::kStageBytes);
            } else {
                const uint32_t leader_full = mapa_shared(smem_u32(&full_bar[stage]), 0);
                a_pair = b_pair = true;
                bar_a = bar_b = leader_full;
            }
            if (C::A_MN && args.a_mn3d) {
                // one copy of all kBM / kMNBox boxes: the map's third
                // dimension walks the MN blocks (see make_map_mn3d)
                if (a_pair) tma_load_3d_pair(pA, bar_a, sa, 0, k0, a_row / C::kMNBox);
                else tma_load_3d(pA, &full_bar[stage], sa, 0, k0, a_row / C::kMNBox);
            } else if (C::A_MN) {
#pragma unroll
                for (int j = 0; j < kBM / C::kMNBox; ++j) {
                    if (a_pair) tma_load_2d_pair(pA, bar_a, sa + j * C::kMNBoxBytes, a_row + C::kMNBox * j, k0);
                    else tma_load_2d(pA, &full_bar[stage], sa + j * C::kMNBoxBytes, a_row + C::kMNBox * j, k0);
                }
            } else {
                if (a_pair) tma_load_2d_pair(pA, bar_a, sa, k0, a_row);
                else tma_load_2d(pA, &full_bar[stage], sa, k0, a_row);
            }
            if (C::B_MN && args.b_mn3d) {
                if (b_pair) tma_load_3d_pair(pB, bar_b, sb, 0, k0 + bk, b_row / C::kMNBox);
                else tma_load_3d(pB, &full_bar[stage], sb, 0, k0 + bk, b_row / C::kMNBox);
            } else if (C::B_MN) {
#pragma unroll
                for (int j = 0; j < C::kBRows / C::kMNBox; ++j) {
                    if (b_pair) tma_load_2d_pair(pB, bar_b, sb + j * C::kMNBoxBytes, b_row + C::kMNBox * j, k0 + bk);
                    else tma_load_2d(pB, &full_bar[stage], sb + j * C::kMNBoxBytes, b_row + C::kMNBox * j, k0 + bk);
                }
            } else {
                if (b_pair) tma_load_2d_pair(pB, bar_b, sb, k0, b_row);
                else tma_load_2d(pB, &full_bar[stage], sb, k0, b_row);
            }
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// MMA issuer (one thread of the leader CTA): every segment's k-blocks into a
// TMEM accumulator; `it` counts segments (the accumulator buffer's parity).
template <class C, int S>
__device__ __forceinline__ void mma_run(const GemmArgs &args, const CtaCtx &x, int &stage, uint32_t &phase,
                                        int &it) {
    uint8_t *stages = x.stages, *staging = x.staging, *aux_smem = x.aux_smem;
    uint64_t *full_bar = x.full_bar, *empty_bar = x.empty_bar, *accf_bar = x.accf_bar, *acce_bar = x.acce_bar,
             *aux_bar = x.aux_bar, *consumed_bar = x.consumed_bar;
    volatile int *abort_flag = x.abort_flag;
    float *rs = x.rs;
    const uint32_t tmem_base = x.tmem_base, rank = x.rank;
    const bool leader = x.leader;
    const int worker = x.worker, slot = x.slot, warp = x.warp, lane = x.lane;
    (void)stages; (void)staging; (void)aux_smem; (void)full_bar; (void)empty_bar; (void)accf_bar;
    (void)acce_bar; (void)aux_bar; (void)consumed_bar; (void)abort_flag; (void)rs; (void)tmem_base;
    (void)rank; (void)leader; (void)worker; (void)slot; (void)warp; (void)lane;
    SegIter si = seg_begin<C::kTileM>(args, worker);
    Seg w;
    for (; seg_next<C::BN, C::kTileM, C::kBKe>(args, si, w); ++it) {
        const int buf = C::kAccBufs == 2 ? (it & 1) : 0;
        const uint32_t aph = C::kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
        if (!mbar_wait(&acce_bar[buf], aph ^ 1u, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * C::BN;
        bool failed = false;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
                failed = true;
                break;
            }
            tc_fence_after_sync();
            const uint32_t a_addr = smem_u32(stages + stage * C::kStageBytes);
            const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
            for (int kk = 0; kk < C::kBKe / C::kUmmaKe; ++kk) {
                // K-major: the next 32 bytes of each row; MN-major: the next
                // kUmmaKe rows of 128 bytes
                const uint32_t mn_step = static_cast<uint32_t>(C::kUmmaKe * 128);
                const uint64_t ad = C::A_MN ? smem_desc_sw128(a_addr + kk * mn_step, C::kMNBoxBytes, 1024)
                                            : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                const uint64_t bd = C::B_MN ? smem_desc_sw128(b_addr + kk * mn_step, C::kMNBoxBytes, 1024)
                                            : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
                const uint32_t acc = (kb > w.kb0 || kk > 0) ? 1u : 0u;
                if (C::F8) {
                    if (C::PAIR) umma_e4m3_pair(d_tmem, ad, bd, C::kIdesc, acc);
                    else umma_e4m3(d_tmem, ad, bd, C::kIdesc, acc);
                } else {
                    if (C::PAIR) umma_bf16_pair(d_tmem, ad, bd, C::kIdesc, acc);
                    else umma_bf16(d_tmem, ad, bd, C::kIdesc, acc);
                }
            }
            // the stage is reusable (in both CTAs) once these MMAs finish
            // (and, in-GEMM RMSNorm, once the norm warps have read its x)
            if (C::PAIR) umma_commit_pair(&empty_bar[stage], 3);
            else umma_commit(&empty_bar[stage]);
            if (C::kNorm) {
                if (C::PAIR) umma_commit_pair(&consumed_bar[stage], 3);
                else umma_commit(&consumed_bar[stage]);
            }
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (failed) break;
        // accumulator ready for the epilogue(s)
        if (C::PAIR) umma_commit_pair(&accf_bar[buf], 3);
        else umma_commit(&accf_bar[buf]);
    }
}

// Epilogue warp: every segment's accumulator out of TMEM, through the fused
// epilogue, to global memory; `it` and `aux_phase` carry over between calls.
template <class C, int S>
__device__ __forceinline__ void epilogue_run(const CUtensorMap *pC0, const CUtensorMap *pC1,
                                             const CUtensorMap *pAux, const GemmArgs &args, const CtaCtx &x,
                                             int &it, uint32_t &aux_phase) {
    uint8_t *stages = x.stages, *staging = x.staging, *aux_smem = x.aux_smem;
    uint64_t *full_bar = x.full_bar, *empty_bar = x.empty_bar, *accf_bar = x.accf_bar, *acce_bar = x.acce_bar,
             *aux_bar = x.aux_bar, *consumed_bar = x.consumed_bar;
    volatile int *abort_flag = x.abort_flag;
    float *rs = x.rs;
    const uint32_t tmem_base = x.tmem_base, rank = x.rank;
    const bool leader = x.leader;
    const int worker = x.worker, slot = x.slot, warp = x.warp, lane = x.lane;
    (void)stages; (void)staging; (void)aux_smem; (void)full_bar; (void)empty_bar; (void)accf_bar;
    (void)acce_bar; (void)aux_bar; (void)consumed_bar; (void)abort_flag; (void)rs; (void)tmem_base;
    (void)rank; (void)leader; (void)worker; (void)slot; (void)warp; (void)lane;
    const int q = warp & 3;                // TMEM lane quarter of this warp
    const int ew = warp - 2;               // epilogue warp index
    // this warp's chunks of a tile: all of them, or its half of them
    const int c_lo = C::kEpiWarps == 8 ? ((ew >> 2) * C::kNumChunks) / 2 : 0;
    const int c_hi = C::kEpiWarps == 8 ? (((ew >> 2) + 1) * C::kNumChunks) / 2 : C::kNumChunks;
    const int row_in_tile = 32 * q + lane;
    const uint32_t leader_acce0 = C::PAIR ? mapa_shared(smem_u32(&acce_bar[0]), 0) : 0u;
    uint8_t *aux_w = aux_smem + q * C::kNumChunks * 4096;  // this warp's 32 rows
    constexpr int kUnits = C::BN / 32;  // 32-column units of a partial-slot row
    constexpr int kSlotsPerWorker = C::PAIR ? 2 : 1;
    // This warp's part of stream-K partial slot `sl`: 32-column unit u, vector
    // j, lane -> float4 ((q * kUnits + u) * 8 + j) * 32 + lane, so that every
    // warp-wide access is 512 contiguous bytes.
    auto part_ptr = [&](int sl, int u, int j) {
        return args.sk_partial + static_cast<size_t>(sl) * kSkSlotFloats +
               ((static_cast<size_t>(q * kUnits + u) * 8 + j) * 32 + lane) * 4;
    };
    // The next segment's operands of this warp (its 32 rows of x or h into
    // shared memory by TMA, its rows' rstd into a register) are fetched as
    // soon as the current segment no longer needs them, so their latency
    // overlaps the main loop instead of the epilogue.  A segment that only
    // writes a partial sum needs neither.
    bool aux_pending = false;  // a prefetch copy issued and not yet waited for
    auto prefetch = [&](const Seg &wn, float &rsc_next) {
        const int r0 = wn.m0 + static_cast<int>(rank) * kBM + 32 * q;
        if (C::kRowScale)
            rsc_next = args.rstd_in ? ((r0 + lane < args.M) ? args.rstd_in[r0 + lane] : 0.0f) : 1.0f;
        if (C::kAux && wn.kb0 == 0 && lane == 0) {
            int nch = 0;
            for (int c = c_lo; c < c_hi; ++c)
                if (wn.n0 + c * C::kChunkCols < args.N) ++nch;
            mbar_arrive_expect_tx(&aux_bar[ew], nch * 4096);
            aux_pending = true;
            for (int c = c_lo; c < c_lo + nch; ++c)
                tma_load_2d(pAux, &aux_bar[ew], aux_w + c * 4096, wn.n0 + c * C::kChunkCols, r0);
        }
    };
    int sbuf = 0;
    float rsc_pre = 1.0f;
    // max |output| of this thread's a (W1) or dh (dgrad-h) values, as stored in bf16
    constexpr bool kAmaxEpi = C::kReluSq || C::EPI == kEpiDgradH;
    const bool want_amax = kAmaxEpi && args.amax_out != nullptr;
    float amax_t = 0.0f;
    const float deq = C::F8 ? (args.deq_a ? *args.deq_a : 1.0f) * (args.deq_b ? *args.deq_b : 1.0f) : 1.0f;
    SegIter si = seg_begin<C::kTileM>(args, worker);
    Seg w;
    bool have = seg_next<C::BN, C::kTileM, C::kBKe>(args, si, w);
    if (have) prefetch(w, rsc_pre);
    for (; have; ++it) {
        // The fused epilogues are nonlinear in the sum over k, so a tile split
        // between workers is finished by the worker holding its first k-blocks
        // (in its last segment); the others (in their first segment) leave
        // fp32 partial sums, which it adds before the fused math.  Reduce
        // epilogues are linear: every segment adds into the output as it is
        // (or, overwriting, a tile that one worker sums whole is stored).
        const bool head = w.kb0 == 0;
        const bool to_partial = !C::kReduce && !head;
        const bool fixup = !C::kReduce && head && w.kb1 < args.k_blocks;
        // a reduce segment adds into C, unless the GEMM overwrites C and this is
        // a tile one worker sums whole (its region was not cleared)
        const bool lin =
            C::kReduce && (!args.overwrite || (args.grp_mode != kGroupK && w.tile >= args.dp_tiles));
        const int m0 = w.m0 + static_cast<int>(rank) * kBM;  // this CTA's rows
        const int buf = C::kAccBufs == 2 ? (it & 1) : 0;
        const uint32_t aph = C::kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
        bool ok = mbar_wait(&accf_bar[buf], aph, abort_flag);
        if (C::kAux && head && ok) {
            ok = mbar_wait(&aux_bar[ew], aux_phase, abort_flag);
            if (ok) {
                aux_pending = false;
                aux_phase ^= 1u;
            }
        }
        // a split tile's contributors: the next workers whose ranges start in it
        int cw_end = worker + 1;
        if (fixup) {
            const int tile_end = (w.tile - si.dp_tiles + 1) * args.k_blocks;
            while (cw_end < args.workers && sk_begin(si, cw_end) < tile_end) ++cw_end;
            for (int cw = worker + 1; cw < cw_end && ok; ++cw)
                ok = flag_wait(&args.sk_flags[(cw * kSlotsPerWorker + static_cast<int>(rank)) * kMaxEpiWarps + ew],
                               abort_flag);
            // The first contributor's partial (this warp's units, 4 KB each) comes
            // into the pipeline stages with one bulk copy: this is the worker's
            // last segment, and its MMAs, which read the stages, have completed.
            constexpr int kCU = C::kChunkCols / 32;
            const int u_lo = c_lo * kCU, nu = (c_hi - c_lo) * kCU;
            if (ok && lane == 0) {
                fence_proxy_async_global();
                mbar_arrive_expect_tx(&aux_bar[ew], nu * 4096);
                bulk_copy_g2s(stages + (q * kUnits + u_lo) * 4096,
                              part_ptr((worker + 1) * kSlotsPerWorker + static_cast<int>(rank), u_lo, 0) - lane * 4,
                              nu * 4096, &aux_bar[ew]);
            }
            if (ok) {
                ok = mbar_wait(&aux_bar[ew], aux_phase, abort_flag);
                if (ok) aux_phase ^= 1u;
            }
        }
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after_sync();
        const bool warp_rows = (m0 + 32 * q) < args.M;
        float rsc = 1.0f;
        if (C::EPI == kEpiFwdW1) rsc = rs[buf * 128 + row_in_tile];
        if (C::kRowScale) rsc = rsc_pre;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * C::BN;

#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
            const int col0 = w.n0 + c * C::kChunkCols;
            if (col0 >= args.N) break;
            constexpr int kChunkUnits = C::kChunkCols / 32;
            float v0[32], v1[32];
            if (C::kOutBf16) tmem_load_64cols(t_row + c * C::kChunkCols, v0, v1);
            else tmem_load_32cols(t_row + c * C::kChunkCols, v0);
            if (to_partial) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    st_global_v4(part_ptr(slot, c * kChunkUnits, j), v0[4 * j], v0[4 * j + 1],
                                 v0[4 * j + 2], v0[4 * j + 3]);
                    if (kChunkUnits == 2)
                        st_global_v4(part_ptr(slot, c * kChunkUnits + 1, j), v1[4 * j], v1[4 * j + 1],
                                     v1[4 * j + 2], v1[4 * j + 3]);
                }
                continue;
            }
            if (fixup) {
                const uint32_t ps = smem_u32(stages + q * kUnits * 4096) + lane * 16;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 p = ld_shared_v4(ps + ((c * kChunkUnits) * 8 + j) * 512);
                    v0[4 * j] += __uint_as_float(p.x); v0[4 * j + 1] += __uint_as_float(p.y);
                    v0[4 * j + 2] += __uint_as_float(p.z); v0[4 * j + 3] += __uint_as_float(p.w);
                    if (kChunkUnits == 2) {
                        const uint4 p1 = ld_shared_v4(ps + ((c * kChunkUnits + 1) * 8 + j) * 512);
                        v1[4 * j] += __uint_as_float(p1.x); v1[4 * j + 1] += __uint_as_float(p1.y);
                        v1[4 * j + 2] += __uint_as_float(p1.z); v1[4 * j + 3] += __uint_as_float(p1.w);
                    }
                }
                // further contributors (ranges shorter than a tile): from L2
                for (int cw = worker + 2; cw < cw_end; ++cw) {
                    const int sl = cw * kSlotsPerWorker + static_cast<int>(rank);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 p = ld_global_cg_v4(part_ptr(sl, c * kChunkUnits, j));
                        v0[4 * j] += p.x; v0[4 * j + 1] += p.y; v0[4 * j + 2] += p.z; v0[4 * j + 3] += p.w;
                        if (kChunkUnits == 2) {
                            const float4 p1 = ld_global_cg_v4(part_ptr(sl, c * kChunkUnits + 1, j));
                            v1[4 * j] += p1.x; v1[4 * j + 1] += p1.y; v1[4 * j + 2] += p1.z; v1[4 * j + 3] += p1.w;
                        }
                    }
                }
            }
            if (C::F8) {
                // E4M3 operands: the dequantisation scales of A and B
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v0[i] *= deq;
                    if (kChunkUnits == 2) v1[i] *= deq;
                }
            }
            // the fused epilogues' [M][N] operand: this row's 64 values of the
            // chunk, from the swizzled shared copy (zero beyond M and N)
            uint4 aux[8];
            if (C::kAux) {
                const uint32_t arow = smem_u32(aux_w + c * 4096) + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    aux[j] = ld_shared_v4(arow + ((static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7)) << 4));
            }
            float cs[32];
            if (C::kColScale) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 g = make_uint4(0, 0, 0, 0);
                    if (col0 + 8 * j < args.N) g = ld_global_nc_v4(args.colscale + col0 + 8 * j);
                    cs[8 * j + 0] = bf16_lo(g.x); cs[8 * j + 1] = bf16_hi(g.x);
                    cs[8 * j + 2] = bf16_lo(g.y); cs[8 * j + 3] = bf16_hi(g.y);
                    cs[8 * j + 4] = bf16_lo(g.z); cs[8 * j + 5] = bf16_hi(g.z);
                    cs[8 * j + 6] = bf16_lo(g.w); cs[8 * j + 7] = bf16_hi(g.w);
                }
            }

            // the staging buffer written kStagingBufs chunks ago must have been
            // read by its TMA store (in-place staging: this chunk's operand copy,
            // already in registers, is not stored from before this tile ends)
            if (!C::kAux) {
                if (lane == 0) bulk_wait_group_read<C::kStagingBufs - 1>();
                __syncwarp();
            }
            uint8_t *st0 = C::kAux ? aux_w + c * 4096
                                   : staging + ((ew * C::kNumOut + 0) * C::kStagingBufs + sbuf) * 4096;
            uint8_t *st1 = C::kAux ? st0
                                   : staging + ((ew * C::kNumOut + (C::kNumOut - 1)) * C::kStagingBufs + sbuf) * 4096;
            const uint32_t s0 = smem_u32(st0) + lane * 128;
            const uint32_t s1 = smem_u32(st1) + lane * 128;
            const uint32_t sw = static_cast<uint32_t>(lane & 7);

            if (C::kOutBf16) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = (j < 4) ? v0[8 * j + i] : v1[8 * (j - 4) + i];
                    uint32_t o[4], o2[4];
                    if (C::kReluSq) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float h0 = rsc * e[2 * i], h1 = rsc * e[2 * i + 1];
                            const float r0 = h0 > 0.0f ? h0 : 0.0f, r1 = h1 > 0.0f ? h1 : 0.0f;
                            if (C::kAOnly) {
                                o[i] = pack_bf16x2(r0 * r0, r1 * r1);
                            } else {
                                o[i] = pack_bf16x2(h0, h1);
                                o2[i] = pack_bf16x2(r0 * r0, r1 * r1);
                            }
                        }
                        if (want_amax)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint32_t av = C::kAOnly ? o[i] : o2[i];
                                amax_t = fmaxf(amax_t, fmaxf(bf16_lo(av), bf16_hi(av)));  // a >= 0
                            }
                    } else if (C::EPI == kEpiStoreBf16) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(rsc * e[2 * i], rsc * e[2 * i + 1]);
                    } else if (C::EPI == kEpiFwdW2) {
                        const uint32_t xs[4] = {aux[j].x, aux[j].y, aux[j].z, aux[j].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            o[i] = pack_bf16x2(bf16_lo(xs[i]) + e[2 * i], bf16_hi(xs[i]) + e[2 * i + 1]);
                    } else {  // kEpiDgradH
                        const uint32_t hs[4] = {aux[j].x, aux[j].y, aux[j].z, aux[j].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float g0 = bf16_lo(hs[i]), g1 = bf16_hi(hs[i]);
                            const float d0 = g0 > 0.0f ? rsc * e[2 * i] * (2.0f * g0) : 0.0f;
                            const float d1 = g1 > 0.0f ? rsc * e[2 * i + 1] * (2.0f * g1) : 0.0f;
                            o[i] = pack_bf16x2(d0, d1);
                            if (want_amax)
                                amax_t = fmaxf(amax_t, fmaxf(fabsf(bf16_lo(o[i])), fabsf(bf16_hi(o[i]))));
                        }
                    }
                    const uint32_t off = ((static_cast<uint32_t>(j) ^ sw) << 4);
                    st_shared_v4(s0 + off, o[0], o[1], o[2], o[3]);
                    if (C::kNumOut == 2) st_shared_v4(s1 + off, o2[0], o2[1], o2[2], o2[3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float e[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        e[i] = v0[4 * j + i];
                        if (C::kColScale) e[i] *= cs[4 * j + i];
                        if (C::EPI == kEpiStoreF32) e[i] *= rsc;
                    }
                    const uint32_t off = ((static_cast<uint32_t>(j) ^ sw) << 4);
                    st_shared_v4(s0 + off, __float_as_uint(e[0]), __float_as_uint(e[1]),
                                 __float_as_uint(e[2]), __float_as_uint(e[3]));
                }
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                if (warp_rows) {
                    const int r0 = m0 + 32 * q + w.crow;
                    if (lin) {
                        tma_reduce_add_2d(pC0, st0, col0, r0);
                    } else {
                        tma_store_2d(pC0, st0, col0, r0);
                        if (C::kNumOut == 2) tma_store_2d(pC1, st1, col0, r0);
                    }
                }
                bulk_commit_group();
            }
            sbuf = C::kStagingBufs == 2 ? sbuf ^ 1 : 0;
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            // TMEM buffer free again (every tcgen05.ld of it has completed)
            mbar_arrive_relaxed(&acce_bar[buf]);
            if (C::PAIR && !leader) mbar_arrive_cluster_relaxed(leader_acce0 + buf * 8);
            // in-place staging: the stores must have read the operand buffers
            // before the next segment's operands are loaded into them
            if (C::kAux) bulk_wait_group_read<0>();
        }
        if (to_partial) {
            // every lane's partial stores are visible before the flag is (after
            // the TMEM release, so the main loop does not wait for the stores)
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(&args.sk_flags[slot * kMaxEpiWarps + ew], 1);
        }
        // every lane is done with this segment's shared operand copy
        have = seg_next<C::BN, C::kTileM, C::kBKe>(args, si, w);
        if (have) prefetch(w, rsc_pre);
    }
    if (lane == 0) {
        bulk_wait_group<0>();
        if (C::kAux && aux_pending) mbar_drain(&aux_bar[ew], aux_phase);
    }
    if (want_amax) {
        // one maximum per epilogue warp; CTA 0 zeroes the slots no CTA holds
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax_t = fmaxf(amax_t, __shfl_xor_sync(0xffffffffu, amax_t, o));
        if (lane == 0) args.amax_out[slot * kMaxEpiWarps + ew] = amax_t;
        if (blockIdx.x == 0) {
            // every slot no epilogue warp writes: the unused warps of each CTA and the CTAs not launched
            for (int i = ew * 32 + lane; i < kMaxSkSlots * kMaxEpiWarps; i += C::kEpiWarps * 32)
                if (i >= static_cast<int>(gridDim.x) * kMaxEpiWarps || i % kMaxEpiWarps >= C::kEpiWarps)
                    args.amax_out[i] = 0.0f;
        }
    }
    __syncwarp();
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
               const __grid_constant__ CUtensorMap tmAux, const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *stages = smem;
    uint8_t *staging = smem + C::kStages * C::kStageBytes;
    uint8_t *aux_smem = staging + C::kStagingBytes;  // [4 warps][chunks][32 rows][128 B]
    uint8_t *ctrl = aux_smem + C::kAuxBytes;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(ctrl);
    uint64_t *empty_bar = full_bar + C::kStages;
    uint64_t *accf_bar = empty_bar + C::kStages;
    uint64_t *acce_bar = accf_bar + 2;
    uint64_t *aux_bar = acce_bar + 2;  // one per epilogue warp
    // in-GEMM RMSNorm: stage s's MMAs have completed, so its x tile may be read
    // by the norm warps (who then release the stage to the producer)
    uint64_t *consumed_bar = aux_bar + kMaxEpiWarps;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 512);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 516);
    float *rs = reinterpret_cast<float *>(ctrl + 1024);  // [2][128], forward W1 only

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kNormArrivals = C::kNorm ? 4u : 0u;
    // pair mode: rank in the CTA pair, the pair's index and count
    const uint32_t rank = C::PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int worker = C::PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int slot = static_cast<int>(blockIdx.x);  // this CTA's stream-K partial slot

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1 + kNormArrivals);
            if (C::kNorm) mbar_init(&consumed_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1 + kNormArrivals);
            // the leader's MMA reuses a TMEM buffer once both CTAs' epilogues drained it
            mbar_init(&acce_bar[b], (C::PAIR && leader) ? 2 * C::kEpiWarps : C::kEpiWarps);
        }
        for (int w = 0; w < C::kEpiWarps; ++w) mbar_init(&aux_bar[w], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC0);
        if (C::kNumOut == 2) prefetch_tensormap(&tmC1);
        if (C::kAux) prefetch_tensormap(&tmAux);
    }
    if (C::PAIR) cluster_sync();  // the peer's barriers exist before anyone signals them
    if (warp == 1) {
        if (C::PAIR) {
            tmem_alloc_pair(tmem_slot, C::kTmemCols);
            tmem_relinquish_alloc_permit_pair();
        } else {
            tmem_alloc(tmem_slot, C::kTmemCols);
            tmem_relinquish_alloc_permit();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel's tail; operands and outputs
    // are touched only after it has completed (a deferred GEMM touches nothing
    // the previous kernel writes, and waits for it at the end instead)
    if (args.pdl != kPdlWaitFirst) griddep_launch_dependents();
    if (args.pdl != kPdlDeferWait) griddep_wait();
    // the next GEMM's stream-K flags start from zero (it runs after this one)
    if (blockIdx.x == 0 && warp == 0 && args.zero_flags)
        for (int i = lane; i < kSkFlagsPerSet; i += 32) args.zero_flags[i] = 0;
    if (args.pdl == kPdlWaitFirst) {
        // the successor may start before this kernel ends and not wait for it:
        // the cleared flags are visible before it can launch
        __threadfence();
        __syncthreads();
        griddep_launch_dependents();
    }

    const CtaCtx x = {stages, staging, aux_smem, full_bar, empty_bar, accf_bar, acce_bar, aux_bar, consumed_bar,
                      abort_flag, rs, tmem_base, rank, leader, worker, slot, warp, lane};
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && !args.skip_loads) {
            int stage = 0;
            uint32_t phase = 0;
            producer_run<C, C::kStages>(&tmA, &tmB, args, x, stage, phase);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            mma_run<C, C::kStages>(args, x, stage, phase, it);
        }
        __syncwarp();
    } else if (warp < 2 + C::kEpiWarps) {
        // --------------------------------------------------------- epilogue
        int it = 0;
        uint32_t aux_phase = 0;
        epilogue_run<C, C::kStages>(&tmC0, &tmC1, &tmAux, args, x, it, aux_phase);
    } else if (C::kSide) {
        // ------------------------------- RMSNorm backward rows (side warps)
        // dn_s is the previous kernel's output: these warps wait for it, while
        // the GEMM's own warps (whose operands it does not write) run on
        side_norm_rows(args.side, warp - 2 - C::kEpiWarps, abort_flag);
    } else if (C::kNorm) {
        // ------------------------------------------- RMSNorm prologue (fwd W1)
        const int r = 32 * (warp - 6) + lane;  // row of this CTA's 128 rows
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        SegIter si = seg_begin<C::kTileM>(args, worker);  // whole tiles only (no stream-K)
        Seg w;
        for (; seg_next<C::BN, C::kTileM, C::kBKe>(args, si, w); ++it) {
            const int m0 = w.m0 + static_cast<int>(rank) * kBM;
            const int buf = C::kAccBufs == 2 ? (it & 1) : 0;
            const uint32_t aph = C::kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
            float ss = 0.0f;
            bool ok = true;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                // the x tile is read after the MMAs that used it completed (they
                // read it from this CTA's shared memory, in pair mode too); the
                // producer refills the stage once these reads are done
                ok = mbar_wait(&consumed_bar[stage], phase, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
                const uint32_t rowaddr = smem_u32(stages + stage * C::kStageBytes) + r * 128;
#pragma unroll
                for (int cidx = 0; cidx < 8; ++cidx)
                    ss += sumsq_bf16x8(ld_shared_v4(rowaddr + ((static_cast<uint32_t>(cidx) ^ sw) << 4)));
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[stage]);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            ok = mbar_wait(&acce_bar[buf], aph ^ 1u, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            const float rstd = 1.0f / sqrtf(ss * args.inv_k + args.eps);
            rs[buf * 128 + r] = rstd;
            const int row = m0 + r;
            if (w.n_blk == 0 && row < args.M) args.rstd_out[row] = rstd;
            __syncwarp();
            if (lane == 0) mbar_arrive(&accf_bar[buf]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (C::PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs may touch it
    if (warp == 1) {
        tc_fence_after_sync();
        if (C::PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else tmem_dealloc(tmem_base, C::kTmemCols);
    }
    // a deferred GEMM completes only after its predecessor has
    if (args.pdl == kPdlDeferWait) griddep_wait();
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Element types of the tensor maps.
enum MapType : int { kMapBf16 = 0, kMapF32 = 1, kMapU8 = 2 };

// 2-D tensor map of a row-major array [outer][inner] with 128-byte swizzle.
inline bool make_map_2d(CUtensorMap *m, const void *ptr, int type, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const uint64_t esz = type == kMapF32 ? 4 : (type == kMapU8 ? 1 : 2);
    const CUtensorMapDataType dt = type == kMapF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : (type == kMapU8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An MN-major operand stored [K][MN] (MN contiguous) as a 3-D map: (kMNBox
// values of MN) x K x (MN / kMNBox blocks), box kMNBox x box_k x nblk.  One copy
// then fills nblk consecutive 128-byte-swizzled boxes of box_k rows, the same
// shared-memory layout as nblk 2-D copies, with one TMA instruction instead of
// nblk (the producer's issue time per k-block halves).  The blocks' stride (the
// box's row, 128 bytes) is below the K stride: the map walks the array in a
// permuted order.  Needs MN a multiple of kMNBox (no partial block).
inline bool make_map_mn3d(CUtensorMap *m, const void *ptr, int type, uint64_t mn, uint64_t k,
                          uint32_t box_mn, uint32_t box_k, uint32_t nblk) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || mn % box_mn != 0) return false;
    const uint64_t esz = type == kMapU8 ? 1 : 2;
    const CUtensorMapDataType dt = type == kMapU8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {box_mn, k, mn / box_mn};
    cuuint64_t strides[2] = {mn * esz, box_mn * esz};
    cuuint32_t box[3] = {box_mn, box_k, nblk};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MLPBLK_SUBSPLIT=0 keeps stream-K ranges for the reduce GEMMs' last round.
inline bool sub_split_enabled() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_SUBSPLIT");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

// MLPBLK_MN3D=0 loads MN-major operands box by box (2-D copies) everywhere.
inline bool mn3d_enabled() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_MN3D");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

// Stream-K scheduling is used unless MLPBLK_STREAMK=0 (whole tiles only);
// MLPBLK_STREAMK=2 takes it wherever the tiles do not fill whole rounds.
inline int streamk_mode() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_STREAMK");
        v = (e && e[0] == '0') ? 0 : ((e && e[0] == '2') ? 2 : 1);
    }
    return v;
}
inline bool streamk_enabled() { return streamk_mode() != 0; }

// M tiles per raster group: MLPBLK_GROUP_M (1..64) when set.  Otherwise 8 when an
// A panel (a tile's rows over all of K) is over 2 MB: a round of 76 pair tiles then
// spans ~8 M-tiles x ~10 N-tiles, about the fewest panels per round, which matters
// once a round's panels no longer fit L2 (the large block's K = 8192 and 16384
// GEMMs re-read 9-12 % less and the power-capped step ran 1.1-1.5 % faster than
// with 16).  With smaller panels 16: a group's A panels stay in L2 across its
// rounds, so B is streamed half as often (the K = 4096 GEMMs read ~10 % less).
inline int raster_group_m(int64_t a_panel_bytes) {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_GROUP_M");
        const int g = e ? atoi(e) : 0;
        v = (g >= 1 && g <= 64) ? g : 0;
    }
    if (v > 0) return v;
    return a_panel_bytes > (2ll << 20) ? 8 : 16;
}

// Builds the tensor maps and launches one GEMM of configuration C.  Pair mode
// launches clusters of two CTAs, one pair per two SMs.
// The tensor maps of one GEMM of configuration C (sets a.a_mn3d, a.b_mn3d).
template <class C>
bool build_maps(int M, int N, int K, const void *A, const void *B, void *C0, void *C1, GemmArgs &a,
                CUtensorMap &mA, CUtensorMap &mB, CUtensorMap &mC0, CUtensorMap &mC1, CUtensorMap &mAux) {
    bool ok = true;
    // operands: 128-byte box rows (kBKe values of K, or kMNBox values of M / N)
    const int op = C::F8 ? kMapU8 : kMapBf16;
    // MN-major operands whose MN is a whole number of boxes: one 3-D copy per
    // operand and k-block
    a.a_mn3d = C::A_MN && kBM / C::kMNBox > 1 && M % C::kMNBox == 0 && mn3d_enabled() &&
               make_map_mn3d(&mA, A, op, M, K, C::kMNBox, C::kBKe, kBM / C::kMNBox);
    if (!a.a_mn3d)
        ok &= C::A_MN ? make_map_2d(&mA, A, op, M, K, C::kMNBox, C::kBKe)
                      : make_map_2d(&mA, A, op, K, M, C::kBKe, kBM);
    // grouped GEMMs: B holds every expert's slice (M-grouped), C every expert's
    // block (K-grouped)
    const uint64_t groups = a.grp_mode != kGroupNone ? static_cast<uint64_t>(a.grp_count) : 1u;
    const uint64_t b_outer = a.grp_mode == kGroupM ? groups : 1u;
    const uint64_t c_rows = static_cast<uint64_t>(M) * (a.grp_mode == kGroupK ? groups : 1u);
    a.b_mn3d = C::B_MN && C::kBRows / C::kMNBox > 1 && N % C::kMNBox == 0 && mn3d_enabled() &&
               make_map_mn3d(&mB, B, op, N, K * b_outer, C::kMNBox, C::kBKe, C::kBRows / C::kMNBox);
    if (!a.b_mn3d)
        ok &= C::B_MN ? make_map_2d(&mB, B, op, N, K * b_outer, C::kMNBox, C::kBKe)
                      : make_map_2d(&mB, B, op, K, N * b_outer, C::kBKe, C::kBRows);
    if (C::kOutBf16) ok &= make_map_2d(&mC0, C0, kMapBf16, N, c_rows, 64, 32);
    else ok &= make_map_2d(&mC0, C0, kMapF32, N, c_rows, 32, 32);
    if (C::kNumOut == 2) ok &= make_map_2d(&mC1, C1, kMapBf16, N, M, 64, 32);
    else mC1 = mC0;
    // the epilogue's [M][N] operand (row stride N), in the output chunks' boxes
    if (C::kAux) ok &= a.aux != nullptr && a.ld_aux == N && make_map_2d(&mAux, a.aux, kMapBf16, N, M, 64, 32);
    else mAux = mC0;
    return ok;
}

template <class C>
int run_gemm_tc(int M, int N, int K, const void *A, const void *B, void *C0, void *C1,
                GemmArgs a, int num_sms, cudaStream_t stream) {
    CUtensorMap mA, mB, mC0, mC1, mAux;
    if (!build_maps<C>(M, N, K, A, B, C0, C1, a, mA, mB, mC0, mC1, mAux)) return MLPBLK_ECUDA;

    // concurrent tile workers: one CTA (pair) per SM (pair of SMs), at most one
    // stream-K partial slot per CTA
    const int cta_per_worker = C::PAIR ? 2 : 1;
    int slots = (num_sms < kMaxSkSlots ? num_sms : kMaxSkSlots) / cta_per_worker;
    if (slots < 1) slots = 1;
    a.M = M;
    a.N = N;
    a.K = K;
    a.m_tiles = (M + C::kTileM - 1) / C::kTileM;
    a.n_tiles = (N + C::BN - 1) / C::BN;
    a.k_blocks = (K + C::kBKe - 1) / C::kBKe;
    const int tiles = a.m_tiles * a.n_tiles;
    const int kb = a.k_blocks;
    a.tiles = tiles;
    if (a.group_m <= 0) a.group_m = raster_group_m(static_cast<int64_t>(C::kTileM) * K * (C::F8 ? 1 : 2));
    int workers = slots;
    if (a.overwrite && !C::kReduce) return MLPBLK_EINVAL;
    const bool sk = !C::kNorm && !a.whole_tiles && a.grp_mode != kGroupK && streamk_enabled() &&
                    (C::kReduce || (a.sk_partial && a.sk_flags));
    if (a.grp_mode == kGroupM && sk && !a.whole_tiles) {
        // M-grouped, split schedule: computed in the kernel from the device row count
        a.grp_split = 1;
        a.dp_tiles = 0;
        a.sk_base = a.sk_rem = a.sk_total = 0;
    } else if (a.grp_mode != kGroupNone) {
        // grouped: whole tiles dealt round robin over a count the kernel reads
        // from device memory (M-grouped) or over every expert's tiles (K-grouped)
        a.grp_split = 0;
        const int64_t upper = a.grp_mode == kGroupK ? static_cast<int64_t>(tiles) * a.grp_count : tiles;
        if (upper < workers) workers = static_cast<int>(upper > 0 ? upper : 1);
        a.dp_tiles = 0;
        a.sk_base = a.sk_rem = a.sk_total = 0;
    } else if (!sk || tiles % workers == 0) {
        // whole tiles: full rounds dealt round robin, the last tiles one each
        if (tiles < workers) workers = tiles;
        a.dp_tiles = tiles / workers * workers;
        a.sk_base = kb;
        a.sk_rem = 0;
        a.sk_total = (tiles - a.dp_tiles) * kb;
    } else {
        // whole-tile rounds while more than two remain; the last one to two
        // rounds' k-blocks are split evenly, so every worker ends together
        const int full = tiles / workers;
        a.dp_tiles = full >= 2 ? (full - 1) * workers : 0;
        const int iters = (tiles - a.dp_tiles) * kb;
        if (a.dp_tiles == 0 && iters < 4 * workers) workers = (iters + 3) / 4;  // >= ~4 k-blocks each
        a.sk_base = iters / workers;
        a.sk_rem = iters % workers;
        a.sk_total = iters;
    }
    a.sub_parts = 0;
    a.sub_kb = 0;
    const int64_t operand_bytes = (static_cast<int64_t>(M) + N) * K * (C::F8 ? 1 : 2);
    if (C::kReduce && sk && a.grp_mode == kGroupNone && tiles % workers != 0 && operand_bytes > (64ll << 20) &&
        sub_split_enabled()) {
        // the last partial round of tiles in k-parts rather than stream-K ranges:
        // S parts of ceil(kb / S) k-blocks (at least 8), S minimising the parts'
        // rounds ceil(R S / workers) / S
        const int full = tiles / workers, rem = tiles - full * workers;
        int best_s = 1;
        double best = 1e30;
        for (int sp = 1; sp <= 8 && (kb + sp - 1) / sp >= 8; ++sp) {
            const double cost = static_cast<double>((rem * sp + workers - 1) / workers) * ((kb + sp - 1) / sp);
            if (cost < best - 1e-9) {
                best = cost;
                best_s = sp;
            }
        }
        a.dp_tiles = full * workers;
        a.sub_parts = best_s;
        a.sub_kb = (kb + best_s - 1) / best_s;
        a.sk_base = a.sk_rem = a.sk_total = 0;
    }
    a.workers = workers;
    a.tile_m = C::kTileM;
    a.tile_n = C::BN;
    if (a.grid_out) *a.grid_out = cta_per_worker * workers;
    if (a.plan_out) {
        *a.plan_out = a;
        return MLPBLK_OK;
    }

    static int attr_set[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MLPBLK_ECUDA;
    if (!attr_set[dev]) {
        const int rc = cuda_status(cudaFuncSetAttribute(
            gemm_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
        if (rc != MLPBLK_OK) return rc;
        attr_set[dev] = 1;
    }
    if (!C::PAIR)
        return launch_pdl(gemm_tc_kernel<C>, dim3(workers), dim3(C::kThreads), C::kSmemBytes, stream,
                          mA, mB, mC0, mC1, mAux, a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * workers, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cuda_status(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<C>, mA, mB, mC0, mC1, mAux, a));
}

// Tile modes a GEMM can launch with.
enum TileMode : int { kTile128 = 0, kTile192 = 1, kTile256 = 2, kTilePair192 = 3, kTilePair256 = 4 };

// Pair tiles are used when MLPBLK_PAIR_TILES is not "0" (default on).
inline bool pair_tiles_enabled() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_PAIR_TILES");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

// Pair modes a GEMM may use (bit mask).
constexpr int kAllowPair256 = 1;
constexpr int kAllowPair192 = 2;  // only with a K-major B operand

// Tile and schedule choice.  Cost, per worker, in units of one 128 x 128 x 64
// MMA step per SM: k-blocks per worker x the tile's MMA work per SM / the shape's
// efficiency.  The efficiencies are measured ones (k-block time of each shape on
// the 120M-class block, where the k-loop waits on operand data: a 256 x 256 pair
// stages the fewest bytes per MMA).  Whole tiles: ceil(tiles / workers) rounds of
// a tile's k-loop.  Stream-K: the k-blocks spread evenly, plus the split tiles'
// fix-up (flag wait, partial copy; ~3 us, and ~2 us more per extra contributor
// when a worker's range is shorter than a tile), which the fp32 += epilogues do
// not need.  Returns the mode, with kUseStreamK set when stream-K wins.
constexpr int kUseStreamK = 0x100;

inline int choose_tile(int M, int N, int K, bool sk_allowed, bool reduce, int num_sms, int allow_pairs,
                       int elem_bytes = 2) {
    // MLPBLK_TILE=128|192|256|pair|pair192 forces one mode where the GEMM
    // allows it (tests run every mode through the same parity suite); the
    // schedule is still chosen by cost
    static int forced = -2;
    if (forced == -2) {
        const char *e = getenv("MLPBLK_TILE");
        if (!e) forced = -1;
        else if (e[0] == 'p') forced = (e[4] == '1') ? kTilePair192 : kTilePair256;
        else if (e[0] == '1') forced = e[1] == '9' ? kTile192 : kTile128;
        else forced = kTile256;
    }
    if (forced == kTilePair256 && !(allow_pairs & kAllowPair256)) forced = kTile256;
    if (forced == kTilePair192 && !(allow_pairs & kAllowPair192)) forced = kTile192;
    const int64_t kb = (static_cast<int64_t>(K) * elem_bytes + 127) / 128;  // 128-byte k-blocks
    const int64_t operand_bytes = (static_cast<int64_t>(M) + N) * K * elem_bytes;
    constexpr int64_t kL2Budget = 64ll << 20;  // half of the 129 MB L2
    double best = 1e300;
    int choice = kTile128;
    auto consider = [&](int mode, int tile_m, int bn, int cta_per_worker, double shape_eff) {
        if (forced >= 0 && mode != forced) return;
        int workers = (num_sms < kMaxSkSlots ? num_sms : kMaxSkSlots) / cta_per_worker;
        if (workers < 1) workers = 1;
        const int64_t tiles = static_cast<int64_t>((M + tile_m - 1) / tile_m) * ((N + bn - 1) / bn);
        const double unit = static_cast<double>(tile_m / cta_per_worker) * bn / (128.0 * 128.0) / shape_eff;
        const double dp = static_cast<double>((tiles + workers - 1) / workers) * kb * unit;
        if (dp < best) {
            best = dp;
            choice = mode;
        }
        if (!sk_allowed || tiles % workers == 0) return;
        const int64_t per = (tiles * kb + workers - 1) / workers;
        double fix = reduce ? 2.0 : 17.0;
        if (!reduce && per < kb) fix += 10.0 * static_cast<double>((kb + per - 1) / per - 1);
        // The split phase's workers run at unrelated k offsets, so tiles that
        // share operand panels no longer read them from L2 at about the same
        // time: with operands well beyond L2 each split k-block costs ~30% more
        // (DRAM reads of the 4096 x 16384 block's K = 16384 GEMMs: 2.7 GB with
        // the split phase, 1.45 GB with whole tiles only)
        const int64_t full = tiles / workers;
        const int64_t split_tiles = tiles - (full >= 2 ? (full - 1) * workers : 0);
        if (operand_bytes > kL2Budget)
            fix += 0.3 * static_cast<double>(split_tiles * kb) / workers * unit;
        const double sk = static_cast<double>(per) * unit + fix;
        if (sk < best || (streamk_mode() == 2 && (mode == choice || forced >= 0))) {
            best = sk;
            choice = mode | kUseStreamK;
        }
    };
    consider(kTile128, kBM, 128, 1, 0.55);
    consider(kTile192, kBM, 192, 1, 0.76);
    consider(kTile256, kBM, 256, 1, 0.90);
    if (allow_pairs & kAllowPair192) consider(kTilePair192, 2 * kBM, 192, 2, 0.75);
    if (allow_pairs & kAllowPair256) consider(kTilePair256, 2 * kBM, 256, 2, 1.0);
    return choice;
}

}  // namespace mlpblk
