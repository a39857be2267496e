// shared_prefix_kernel.cuh -- decode attention for batches whose sequences
// share prompt-prefix blocks.
//
// Sequences forked from one prompt (parallel sampling, beam search) hold the
// same physical blocks for the prompt and only their own blocks after it
// (Hacker News thread on PagedAttention: blocks of one sequence are shared by
// its siblings; Qualiteg, "About PagedAttention for LLM serving": a block
// table per sequence maps logical onto physical blocks).  Each shared block
// then needs to come from HBM once for the whole group, not once per
// sequence: a "prefix item" stages a block once and multiplies it against
// the query rows of every member (members x GQA group <= 32 rows, two 16-row
// mma.sync tiles; 16 rows, one tile, for 64- and 256-wide heads and for fp32
// pools, whose tiles are TF32 with three products each), while "suffix
// items" walk each sequence's own blocks.
// Every item leaves a normalised partial output and its log2-sum-exp per
// query row (or the final row when it is the sequence's only part); the
// combine pass merges the parts, which is exact for softmax.
//
// Work is a list written by the planning kernel and pulled, one item per
// warp, from an atomic counter by a persistent grid: prefix items first (the
// largest), then suffix items.  A warp runs its item alone, through its own
// ring of TMA stages, so no warp ever waits for another: the slots its last
// blocks free already take the first blocks of its next item (whose entry,
// block ids and partial counts it fetched while the current item streamed),
// and it writes its rows straight from registers while those land.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "decode_kernel.cuh"

namespace pkv {

constexpr int kSpWarps = 4;
// query rows and 16-row accumulator tiles of one item
template <typename T, int D>
constexpr int kSpRows = sp_rows_for(D, (int)sizeof(T));
template <typename T, int D>
constexpr int kSpTiles = kSpRows<T, D> / 16;
// Shared memory per CTA: two CTAs (8 warps) per SM for 128- and 256-wide
// heads, which is what the register budget of their accumulators allows, and
// four CTAs (16 warps) for the one-tile items of a 64-wide head.  Each warp's
// ring takes the stages that fit: two for a 128-wide head, two for a 64-wide
// one, and one 16 KiB stage for a 256-wide head, whose eight warps per SM then
// hide more latency than two stages for four warps would (one CTA per SM).
// fp32 pools (twice the bytes a stage) fit one stage for both head sizes.
template <int D>
constexpr int kSpSmemTarget = D == 64 ? 55 * 1024 : 112 * 1024;

template <typename T, int D, int BS>
struct SpSmem {
    using Gm = Geom<T, D, BS>;
    static constexpr int kQ = kSpRows<T, D> * D * (int)sizeof(T);  // a warp's query rows (swizzled slabs)
    static constexpr int kMisc = 256;
    static constexpr int kFixed = kSpWarps * kQ + kMisc + 1024;
    static constexpr int kStagesFit = (kSpSmemTarget<D> - kFixed) / (kSpWarps * Gm::kStageBytes);
    static constexpr int NST = kStagesFit < 1 ? 1 : (kStagesFit > 8 ? 8 : kStagesFit);
    static constexpr int kRing = kSpWarps * NST * Gm::kStageBytes;
    // a one-stage ring has separate K and V barriers per stage (its K half
    // refills while the V half is waited on and used, and the other way round)
    static constexpr bool kSplitKV = NST == 1;
    static constexpr int kBarsPerWarp = kSplitKV ? 2 * NST : NST;
    static constexpr int kBars = kSpWarps * kBarsPerWarp * 8;
    // offsets from the 1024-aligned base
    static constexpr int oQ = kRing;
    static constexpr int oBars = oQ + kSpWarps * kQ;
    static constexpr int kBytes = oBars + kBars + kMisc + 1024;
};


// 16-byte asynchronous global->shared copy; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// A work item as its warp sees it (fields of SpEntry plus derived values).
struct SpItem {
    int g, seq0, nseq, tbl_seq, b0, b1, slot, tok_end;
    int nb;  // blocks of the item
    int R;   // query rows (nseq * group)
};

// ------------------------------------------------------ tensor-core rows

// Online-softmax attention of up to two 16-row tiles of query rows against
// 16-token sub-blocks of K and V staged in shared memory.  The query tile is
// read from shared memory with ldmatrix (it would not fit in registers next
// to two tiles of accumulators); P is split into a 16-bit high part and a 16-bit
// remainder so the weights keep about 16 bits.
template <typename T, int D, int BS>
struct SpMma {
    using MM = Mma16<T>;
    static constexpr int ND = D / 8;  // n-tiles of O
    static constexpr int NT = kSpTiles<T, D>;
    float o[NT][ND][4];
    // [tile][row gid / gid+8]: m is the row's reference (log2 units), l its
    // lane-partial sum of weights relative to m
    float m[NT][2], l[NT][2];
    int gid, tig;
    bool fresh;  // no block seen yet: the first one sets every row's reference

    __device__ __forceinline__ void reset(int lane) {
        gid = lane >> 2;
        tig = lane & 3;
        fresh = true;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            m[t][0] = m[t][1] = 0.f;
            l[t][0] = l[t][1] = 0.f;
#pragma unroll
            for (int n = 0; n < ND; ++n) o[t][n][0] = o[t][n][1] = o[t][n][2] = o[t][n][3] = 0.f;
        }
    }

    // V rows r0+nvalid .. r0+15 of a partial run may hold stale bits (even
    // NaN, and 0 * NaN is NaN): zero them in the stage before P V reads it.
    // The fence orders these writes before the TMA refill of the slot.
    __device__ __forceinline__ void zero_tail(uint32_t vaddr, int r0, int nvalid, int lane) {
        constexpr int CH = D * 2 / 16;
        for (int q = lane; q < (16 - nvalid) * CH; q += 32)
            sts_zero16(vaddr + swz_offset<BS>(r0 + nvalid + q / CH, q % CH));
        fence_proxy_async_smem();
        __syncwarp();
    }

    // S = Q K^T for tokens r0 .. r0+15 of the staged K block, the first
    // `nvalid` (1..16) of which are context tokens (query tile at qaddr), and
    // the online softmax; P, as a high part and remainder, goes to ph / pl.
    template <int MT, int QR>
    __device__ __forceinline__ void scores(uint32_t kaddr, uint32_t qaddr, int r0, int nvalid,
                                           float scale_log2, int lane, uint32_t (&ph)[MT][4],
                                           uint32_t (&pl)[MT][4]) {
        const bool partial = nvalid < 16;  // the item's last run only (warp-uniform)
        float s[MT][2][4];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[t][nt][0] = s[t][nt][1] = s[t][nt][2] = s[t][nt][3] = 0.f;
        // S = Q K^T, 32 head-dim columns per step
#pragma unroll
        for (int kc = 0; kc < D / 32; ++kc) {
            uint32_t qa[MT][2][4];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int qrow = t * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    ldsm_x4(qaddr + swz_offset<QR>(qrow, (2 * kc + h) * 2 + (lane >> 4)),
                            qa[t][h][0], qa[t][h][1], qa[t][h][2], qa[t][h][3]);
            }
            uint32_t kb[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                ldsm_x4(kaddr + swz_offset<BS>(r0 + nt * 8 + (lane & 7), kc * 4 + (lane >> 3)),
                        kb[nt][0], kb[nt][1], kb[nt][2], kb[nt][3]);
            // consecutive MMAs update different accumulators (no back-to-back chain)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        MM::mma(s[t][nt], qa[t][h], kb[nt][2 * h], kb[nt][2 * h + 1]);
        }
        // Online softmax per row (log2 domain) against a lazy reference: a
        // row's reference m moves, and its sum and accumulators are rescaled,
        // only when one of its scores passes m by more than kLazyLog2.  Until
        // then the weights stay at most 2^kLazyLog2, which the 16-bit high part
        // and remainder of P carry with the same relative precision as weights
        // below 1, and the final division by the row's sum is unchanged
        // (softmax does not depend on the reference subtracted).  Most blocks
        // then skip the row-max shuffles and the multiply of every accumulator;
        // the score scale and the subtraction of m are one fused multiply-add.
        constexpr float kLazyLog2 = 8.f;
        if (partial) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (nt * 8 + 2 * tig + e >= nvalid)
                            s[t][nt][e] = s[t][nt][2 + e] = -CUDART_INF_F;
        }
        bool grow = fresh;
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[t][nt][e] = fmaf(s[t][nt][e], scale_log2, -m[t][0]);
                    s[t][nt][2 + e] = fmaf(s[t][nt][2 + e], scale_log2, -m[t][1]);
                    grow |= s[t][nt][e] > kLazyLog2;
                    grow |= s[t][nt][2 + e] > kLazyLog2;
                }
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        mx0 = fmaxf(mx0, s[t][nt][e]);
                        mx1 = fmaxf(mx1, s[t][nt][2 + e]);
                    }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                // every row has a context token (nvalid >= 1), so mx is finite;
                // the first block takes its maximum, later ones only raise m
                const float d0 = fresh ? mx0 : fmaxf(mx0, 0.f);
                const float d1 = fresh ? mx1 : fmaxf(mx1, 0.f);
                const float a0 = fresh ? 0.f : fast_exp2(-d0);
                const float a1 = fresh ? 0.f : fast_exp2(-d1);
                m[t][0] += d0;
                m[t][1] += d1;
                l[t][0] *= a0;
                l[t][1] *= a1;
#pragma unroll
                for (int n = 0; n < ND; ++n) {
                    o[t][n][0] *= a0;
                    o[t][n][1] *= a0;
                    o[t][n][2] *= a1;
                    o[t][n][3] *= a1;
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[t][nt][e] -= d0;
                        s[t][nt][2 + e] -= d1;
                    }
            }
            fresh = false;
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[t][nt][e] = fast_exp2(s[t][nt][e]);
                    s[t][nt][2 + e] = fast_exp2(s[t][nt][2 + e]);
                    ls0 += s[t][nt][e];
                    ls1 += s[t][nt][2 + e];
                }
            l[t][0] += ls0;
            l[t][1] += ls1;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float *sv = s[t][j];
                ph[t][2 * j] = MM::pack(sv[0], sv[1]);
                ph[t][2 * j + 1] = MM::pack(sv[2], sv[3]);
                pl[t][2 * j] = MM::pack(sv[0] - MM::lo(ph[t][2 * j]), sv[1] - MM::hi(ph[t][2 * j]));
                pl[t][2 * j + 1] =
                    MM::pack(sv[2] - MM::lo(ph[t][2 * j + 1]), sv[3] - MM::hi(ph[t][2 * j + 1]));
            }
        }
    }

    // O += P V for the same tokens of the staged V block (rows past the
    // context zeroed first).
    template <int MT>
    __device__ __forceinline__ void accumulate(uint32_t vaddr, int r0, int lane,
                                               const uint32_t (&ph)[MT][4], const uint32_t (&pl)[MT][4]) {
        const int tok = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int np = 0; np < ND / 2; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vaddr + swz_offset<BS>(tok, np * 2 + (lane >> 4)), b0, b1, b2, b3);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                MM::mma(o[t][2 * np], ph[t], b0, b1);
                MM::mma(o[t][2 * np + 1], ph[t], b2, b3);
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                MM::mma(o[t][2 * np], pl[t], b0, b1);
                MM::mma(o[t][2 * np + 1], pl[t], b2, b3);
            }
        }
    }

    // Both, for tokens r0 .. r0+15 of a block staged whole (K at kaddr, V at
    // vaddr); the stale V rows are zeroed first, so the writes overlap the
    // arithmetic.
    template <int MT, int QR>
    __device__ __forceinline__ void sub_block(uint32_t kaddr, uint32_t vaddr, uint32_t qaddr,
                                              int r0, int nvalid, float scale_log2, int lane) {
        if (nvalid < 16) zero_tail(vaddr, r0, nvalid, lane);
        uint32_t ph[MT][4], pl[MT][4];
        scores<MT, QR>(kaddr, qaddr, r0, nvalid, scale_log2, lane, ph, pl);
        accumulate<MT>(vaddr, r0, lane, ph, pl);
    }

    // query buffer of QR rows (32: two tiles for a prefix item; 16: one warp's own)
    template <int MT, int QR>
    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, uint32_t qaddr, int nvalid,
                                          float scale_log2, int lane) {
#pragma unroll
        for (int h = 0; h < BS / 16; ++h) {
            const int nv = nvalid - h * 16;
            if (nv > 0) sub_block<MT, QR>(kaddr, vaddr, qaddr, h * 16, nv < 16 ? nv : 16, scale_log2, lane);
        }
    }
};

// fp32 storage: one 16-row tile of query rows as m16n8k8 TF32 tiles, each
// product as three TF32 products, each k-step (and each block's P V) from a
// zero accumulator added by rounded fp32 adds, so that scores and outputs
// keep about fp32 accuracy.  Q
// and K fragments come from their swizzled buffers by ldmatrix (an 8-row,
// 16-byte matrix of the 16-bit view is an 8x4 block of fp32, one value a
// lane); P moves from the accumulator layout to the A layout by shuffles in
// each group of four lanes; V fragments come by 16-byte loads, four O
// columns at a time, so that inside each 32-column group column 32g + 4n + j
// is n-tile j's column n.  The online softmax keeps the lazy reference of
// the 16-bit tiles.
template <int D, int BS>
struct SpTf32 {
    static constexpr int KS = D / 8;   // k-steps of the QK^T product
    static constexpr int NG = D / 32;  // 32-column groups of O
    float o[NG][4][4];                 // column group, n-tile, C fragment
    float m[1][2], l[1][2];            // rows gid / gid+8: reference, lane-partial sum
    int gid, tig;
    bool fresh;                        // no block seen yet in this item

    __device__ __forceinline__ void reset(int lane) {
        gid = lane >> 2;
        tig = lane & 3;
        fresh = true;
        m[0][0] = m[0][1] = 0.f;
        l[0][0] = l[0][1] = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[g][j][0] = o[g][j][1] = o[g][j][2] = o[g][j][3] = 0.f;
    }

    // V rows r0+nvalid .. r0+15 of a partial run may hold stale bits (even
    // NaN): zero them in the stage before P V reads it, fenced against the
    // TMA refill of the slot.
    __device__ __forceinline__ void zero_tail(uint32_t vaddr, int r0, int nvalid, int lane) {
        constexpr int CH = D * 4 / 16;
        for (int q = lane; q < (16 - nvalid) * CH; q += 32)
            sts_zero16(vaddr + swz_offset<BS>(r0 + nvalid + q / CH, q % CH));
        fence_proxy_async_smem();
        __syncwarp();
    }

    // S = Q K^T for tokens r0 .. r0+15 (the first nvalid are context tokens)
    // and the online softmax; P for the two 8-token k-steps of P V, as a
    // TF32 high part and remainder in the A layout, goes to ph / pl.
    template <int QR>
    __device__ __forceinline__ void scores(uint32_t kaddr, uint32_t qaddr, int r0, int nvalid,
                                           float scale_log2, int lane, uint32_t (&ph)[2][4],
                                           uint32_t (&pl)[2][4]) {
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        // ldmatrix.x4: lane L names row (L & 7) of matrix L >> 3; for Q the
        // matrices are (rows 0-7 | 8-15) x (columns 8ks..+3 | +4..+7), in the
        // order of the A fragment; for K (tokens 0-7 | 8-15) x the same columns
        const int qrow = ((lane >> 3) & 1) * 8 + (lane & 7), qhalf = lane >> 4;
        const int ktok = r0 + (lane >> 4) * 8 + (lane & 7), khalf = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t q[4], kr[4];
            ldsm_x4(qaddr + swz_offset<QR>(qrow, ks * 2 + qhalf), q[0], q[1], q[2], q[3]);
            ldsm_x4(kaddr + swz_offset<BS>(ktok, ks * 2 + khalf), kr[0], kr[1], kr[2], kr[3]);
            uint32_t ah[4], al[4], kh[4], kl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                tf32_split(__uint_as_float(q[i]), ah[i], al[i]);
                tf32_split(__uint_as_float(kr[i]), kh[i], kl[i]);
            }
            // each k-step from a zero accumulator, added by a rounded fp32 add
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float t[4] = {0.f, 0.f, 0.f, 0.f};
                mma_tf32x3(t, ah, al, kh[2 * nt], kh[2 * nt + 1], kl[2 * nt], kl[2 * nt + 1]);
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] += t[e];
            }
        }
        if (nvalid < 16) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (nt * 8 + 2 * tig + e >= nvalid) s[nt][e] = s[nt][2 + e] = -CUDART_INF_F;
        }
        bool grow = fresh;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = fmaf(s[nt][e], scale_log2, -m[0][0]);
                s[nt][2 + e] = fmaf(s[nt][2 + e], scale_log2, -m[0][1]);
                grow |= s[nt][e] > 8.f;
                grow |= s[nt][2 + e] > 8.f;
            }
        if (__any_sync(0xffffffffu, grow)) {
            float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            // every row has a context token (nvalid >= 1), so mx is finite
            const float d0 = fresh ? mx0 : fmaxf(mx0, 0.f), d1 = fresh ? mx1 : fmaxf(mx1, 0.f);
            const float a0 = fresh ? 0.f : fast_exp2(-d0), a1 = fresh ? 0.f : fast_exp2(-d1);
            m[0][0] += d0;
            m[0][1] += d1;
            l[0][0] *= a0;
            l[0][1] *= a1;
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    o[g][j][0] *= a0;
                    o[g][j][1] *= a0;
                    o[g][j][2] *= a1;
                    o[g][j][3] *= a1;
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] -= d0;
                    s[nt][2 + e] -= d1;
                }
            fresh = false;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[nt][e] = fast_exp2(s[nt][e]);
                l[0][e >> 1] += s[nt][e];
            }
        // C layout (row g, columns 2t, 2t+1) -> A layout (row g, columns t, t+4)
        const int base = lane & ~3, srcA = base + (tig >> 1), srcB = srcA + 2;
        const bool odd = tig & 1;
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            const float x0 = __shfl_sync(0xffffffffu, s[kt][0], srcA);
            const float x1 = __shfl_sync(0xffffffffu, s[kt][1], srcA);
            const float y0 = __shfl_sync(0xffffffffu, s[kt][2], srcA);
            const float y1 = __shfl_sync(0xffffffffu, s[kt][3], srcA);
            const float z0 = __shfl_sync(0xffffffffu, s[kt][0], srcB);
            const float z1 = __shfl_sync(0xffffffffu, s[kt][1], srcB);
            const float w0 = __shfl_sync(0xffffffffu, s[kt][2], srcB);
            const float w1 = __shfl_sync(0xffffffffu, s[kt][3], srcB);
            tf32_split(odd ? x1 : x0, ph[kt][0], pl[kt][0]);  // P[g][t]
            tf32_split(odd ? y1 : y0, ph[kt][1], pl[kt][1]);  // P[g+8][t]
            tf32_split(odd ? z1 : z0, ph[kt][2], pl[kt][2]);  // P[g][t+4]
            tf32_split(odd ? w1 : w0, ph[kt][3], pl[kt][3]);  // P[g+8][t+4]
        }
    }

    // O += P V for the same tokens of the staged V block (rows past the
    // context zeroed first).
    __device__ __forceinline__ void accumulate(uint32_t vaddr, int r0, int lane,
                                               const uint32_t (&ph)[2][4], const uint32_t (&pl)[2][4]) {
        // from zero accumulators, added to O by rounded fp32 adds
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            float f[2][2][4];
#pragma unroll
            for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = lds128(vaddr + swz_offset<BS>(r0 + kt * 8 + tig + 4 * h, g * 8 + gid));
                    f[kt][h][0] = __uint_as_float(v.x);
                    f[kt][h][1] = __uint_as_float(v.y);
                    f[kt][h][2] = __uint_as_float(v.z);
                    f[kt][h][3] = __uint_as_float(v.w);
                }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    uint32_t bh0, bl0, bh1, bl1;
                    tf32_split(f[kt][0][j], bh0, bl0);
                    tf32_split(f[kt][1][j], bh1, bl1);
                    mma_tf32x3(t, ph[kt], pl[kt], bh0, bh1, bl0, bl1);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) o[g][j][e] += t[e];
            }
        }
    }

    // a block staged whole; the stale V rows are zeroed first
    template <int MT, int QR>
    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, uint32_t qaddr, int nvalid,
                                          float scale_log2, int lane) {
#pragma unroll
        for (int h = 0; h < BS / 16; ++h) {
            const int nv = nvalid - h * 16;
            if (nv > 0) {
                const int n = nv < 16 ? nv : 16;
                if (n < 16) zero_tail(vaddr, h * 16, n, lane);
                uint32_t ph[2][4], pl[2][4];
                scores<QR>(kaddr, qaddr, h * 16, n, scale_log2, lane, ph, pl);
                accumulate(vaddr, h * 16, lane, ph, pl);
            }
        }
    }

    // head column of C element e (0, 1) of n-tile j in column group g
    __device__ __forceinline__ int col(int g, int j, int e) const { return g * 32 + 8 * tig + j + 4 * e; }
};

// ------------------------------------------------------------------ kernel

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kSpWarps * 32)
    shared_prefix_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv, const SpArgs a) {
    using Gm = Geom<T, D, BS>;
    using Sm = SpSmem<T, D, BS>;
    constexpr int NST = Sm::NST;
    constexpr int QCH = D * (int)sizeof(T) / 16;  // 16-byte chunks per query row
    constexpr int ND = D / 8;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.num_kv_heads, G = a.group;
    unsigned char *wstage = smem + warp * NST * Gm::kStageBytes;
    constexpr bool kSplit = Sm::kSplitKV;
    static_assert(!kSplit || BS == 16, "split K/V ring: 16-row runs");
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + Sm::oBars) + warp * Sm::kBarsPerWarp;
    const uint32_t qaddr = smem_u32(smem + Sm::oQ + warp * Sm::kQ);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < Sm::kBarsPerWarp; ++i) mbar_init(&wbar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncwarp();
    griddep_wait();  // the work list of the planning kernel is complete and visible
    const bool planned = sp_plan_matches(a);
    if (!planned && blockIdx.x == 0 && threadIdx.x == 0) raise_fault(a.dev_error, PKV_FAULT_PREFIX);
    const int nP = planned ? a.count[0] : 0, nS = planned ? a.count[1] : 0;
    const int totalP = nP * Hkv, total = (nP + nS) * Hkv;

    auto fetch = [&]() -> int {
        int v = 0;
        if (lane == 0) v = atomicAdd(a.counter, 1);
        return __shfl_sync(FULL, v, 0);
    };
    // lane j < 8 holds field j of an item's entry (prefix items, then suffix items)
    auto field = [&](int j) -> int {
        if (j >= total) return 0;
        const int e = j < totalP ? j / Hkv : a.suffix_base + (j - totalP) / Hkv;
        return lane < 8 ? reinterpret_cast<const int *>(a.entries + e)[lane] : 0;
    };
    auto decode = [&](int j, int f) -> SpItem {
        SpItem t;
        t.g = (j < totalP ? j : j - totalP) % Hkv;
        t.seq0 = __shfl_sync(FULL, f, 0);
        t.nseq = __shfl_sync(FULL, f, 1);
        t.tbl_seq = __shfl_sync(FULL, f, 2);
        t.b0 = __shfl_sync(FULL, f, 3);
        t.b1 = __shfl_sync(FULL, f, 4);
        t.slot = __shfl_sync(FULL, f, 5);
        t.tok_end = __shfl_sync(FULL, f, 6);
        t.nb = t.b1 - t.b0;
        t.R = t.nseq * G;
        return t;
    };
    // physical block of the item's i-th run (chunk of 32, one per lane); a
    // block of more than 16 tokens is 2^ushift runs, named by one table entry
    const int ushift = a.unit_shift;
    auto bt_load = [&](const SpItem &t, int chunk) -> int {
        const int i = chunk * 32 + lane;
        if (i >= t.nb) return -1;
        return __ldg(a.block_tables + (size_t)t.tbl_seq * a.max_blocks_per_seq + ((t.b0 + i) >> ushift));
    };
    // partial count of the sequence of row `lane` of the item
    auto nparts_of = [&](const SpItem &t) -> int {
        return lane < t.R ? a.nparts[t.seq0 + lane / G] : 0;
    };
    // stage run `run` (of its sequence) of block pb at absolute ring position k
    const uint64_t kv_policy = l2_evict_first_policy();  // K/V tiles are read once
    // one half (0: K, 1: V) of the stage at ring position k of a split ring,
    // on its own barrier (K barriers first, then V barriers)
    auto issue_half = [&](int h, int g, unsigned k, int pb, int run) {
        if (lane == 0) {
            uint64_t *bar = &wbar[h * NST + k % NST];
            if (pb >= 0 && pb < a.num_blocks) {
                mbar_arrive_expect_tx(bar, Gm::kTileBytes);
                unsigned char *dst = wstage + (k % NST) * Gm::kStageBytes + h * Gm::kTileBytes;
                const int y = (((pb * Hkv + g) << ushift) + (run & ((1 << ushift) - 1))) * BS;
#pragma unroll
                for (int sl = 0; sl < Gm::kSlabs; ++sl)
                    tma_load_2d_hint(dst + sl * Gm::kSlabBytes, h ? &tmv : &tmk, sl * Gm::kSlabElems, y,
                                     bar, kv_policy);
            } else {
                raise_fault(a.dev_error, PKV_FAULT_BLOCK_ID);
                mbar_arrive(bar);
            }
        }
    };
    auto issue = [&](int g, unsigned k, int pb, int run) {
        if constexpr (kSplit) {
            issue_half(0, g, k, pb, run);
            issue_half(1, g, k, pb, run);
            return;
        }
        if (lane == 0) {
            uint64_t *bar = &wbar[k % NST];
            if (pb >= 0 && pb < a.num_blocks) {
                mbar_arrive_expect_tx(bar, Gm::kStageBytes);
                unsigned char *dk = wstage + (k % NST) * Gm::kStageBytes;
                unsigned char *dv = dk + Gm::kTileBytes;
                const int y = (((pb * Hkv + g) << ushift) + (run & ((1 << ushift) - 1))) * BS;
#pragma unroll
                for (int sl = 0; sl < Gm::kSlabs; ++sl) {
                    tma_load_2d_hint(dk + sl * Gm::kSlabBytes, &tmk, sl * Gm::kSlabElems, y, bar, kv_policy);
                    tma_load_2d_hint(dv + sl * Gm::kSlabBytes, &tmv, sl * Gm::kSlabElems, y, bar, kv_policy);
                }
            } else {
                raise_fault(a.dev_error, PKV_FAULT_BLOCK_ID);
                mbar_arrive(bar);
            }
        }
    };
    // the item's query rows into the warp's buffer (zero rows pad the last tile)
    const T *qg = reinterpret_cast<const T *>(a.q);
    auto load_rows = [&](const SpItem &t) {
        const int rows_pad = t.R > 16 ? 32 : 16;
#pragma unroll 2
        for (int idx = lane; idx < rows_pad * QCH; idx += 32) {
            const int r = idx / QCH, c = idx - r * QCH;
            const T *src = qg;
            int bytes = 0;
            if (r < t.R) {
                const int sq = t.seq0 + r / G, h = t.g * G + r % G;
                src = qg + ((size_t)sq * a.num_heads + h) * D + c * (16 / (int)sizeof(T));
                bytes = 16;
            }
            cp_async16(qaddr + swz_offset<kSpRows<T, D>>(r, c), src, bytes);
        }
        cp_async_commit();
    };

    constexpr bool kF32 = sizeof(T) == 4;  // fp32 storage: TF32 tiles
    using Path = std::conditional_t<kF32, SpTf32<D, BS>, SpMma<T, D, BS>>;
    Path path;
    unsigned ctr = 0;  // blocks this warp has consumed (stage ring position, across items)
    int j0 = fetch();
    if (j0 < total) {
        SpItem it = decode(j0, field(j0));
        int np = nparts_of(it);
        int ent0 = bt_load(it, 0), ent1 = bt_load(it, 1);
        // the first stages before the query rows: every warp copies its rows
        // at once here, and the K/V requests should not queue behind them
#pragma unroll 1
        for (int j = 0; j < NST && j < it.nb; ++j) issue(it.g, j, __shfl_sync(FULL, ent0, j), it.b0 + j);
        load_rows(it);
#pragma unroll 1
        for (;;) {
            cp_async_wait_all();
            __syncwarp();  // the item's query rows are in place
            // The next item is claimed as late as its latency allows, so the
            // longest-first list keeps balancing the warps until its end: a
            // long item claims it three blocks before its first stage is due,
            // reads the index a block later and decodes the entry a block
            // after that; a short item claims it now and reads it after its
            // first blocks.  Its first stages go into the ring slots this
            // item frees in its last NST blocks (ring positions continue
            // across items), or after the loop if its block ids came too late.
            const bool late = it.nb > NST + 3;
            const int claim_at = late ? it.nb - NST - 3 : -1;
            const int read_at = late ? claim_at + 1 : 0;
            int jn_raw = 0;
            if (!late && lane == 0) jn_raw = atomicAdd(a.counter, 1);
            int jn = total, fn = 0;
            int entn0 = -1, entn1 = -1, np1 = 0, nx_g = 0, nx_b0 = 0, nx_nb = 0;
            bool known = false;  // the next item's index and entry are decoded
            auto learn_next = [&]() {
                if (jn < total) {
                    const SpItem n1 = decode(jn, fn);
                    entn0 = bt_load(n1, 0);
                    entn1 = bt_load(n1, 1);
                    np1 = nparts_of(n1);
                    nx_g = n1.g;
                    nx_b0 = n1.b0;
                    nx_nb = n1.nb;
                }
                known = true;
            };
            const int learn_at = late ? claim_at + 2 : (it.nb > NST ? 1 : 0);
            const bool two = it.R > 16;
            unsigned issued = ctr + min(NST, it.nb);  // ring positions issued so far
            unsigned issued_k = issued;               // (K halves, for a split ring)
            path.reset(lane);
            int cb = 0;
            bool ok = true;
            auto bt_get = [&](int i) -> int {
                return (i >> 5) == cb ? __shfl_sync(FULL, ent0, i & 31) : __shfl_sync(FULL, ent1, i & 31);
            };
            int i = 0;
#pragma unroll 1
            for (; i < it.nb; ++i) {
                if ((i >> 5) != cb) {
                    cb = i >> 5;
                    ent0 = ent1;
                    ent1 = bt_load(it, cb + 1);
                }
                const int pb = bt_get(i);
                const unsigned kk = ctr + i;
                if constexpr (kSplit) {
                    // K half: scores; then the K half of position kk + NST
                    // (this item's block i + NST, or the next item's block j,
                    // in order) goes into the freed slot while the V half is
                    // waited on and used
                    ok = __all_sync(FULL, mbar_wait(&wbar[kk % NST], (kk / NST) & 1));
                    if (!ok) break;
                    const bool valid = pb >= 0 && pb < a.num_blocks;
                    const int nvalid = min(BS, it.tok_end - (it.b0 + i) * BS);
                    const uint32_t kaddr = smem_u32(wstage + (kk % NST) * Gm::kStageBytes);
                    const uint32_t vaddr = kaddr + Gm::kTileBytes;
                    // P between the scores and P V: two 16-row tiles of 16-bit
                    // pairs, or the two 8-token k-steps of a TF32 tile
                    uint32_t ph[2][4], pl[2][4];
                    auto &ph1 = reinterpret_cast<uint32_t(&)[1][4]>(ph);
                    auto &pl1 = reinterpret_cast<uint32_t(&)[1][4]>(pl);
                    if (valid) {
                        if constexpr (kF32)
                            path.template scores<kSpRows<T, D>>(kaddr, qaddr, 0, nvalid, a.scale_log2, lane, ph, pl);
                        else if (kSpTiles<T, D> == 2 && two)
                            path.template scores<2, kSpRows<T, D>>(kaddr, qaddr, 0, nvalid, a.scale_log2, lane, ph, pl);
                        else
                            path.template scores<1, kSpRows<T, D>>(kaddr, qaddr, 0, nvalid, a.scale_log2, lane, ph1, pl1);
                    }
                    int ng = -1, npb = -1, nrun = 0;
                    if (i + NST < it.nb) {
                        ng = it.g;
                        npb = bt_get(i + NST);
                        nrun = it.b0 + i + NST;
                    } else if (it.nb >= NST && issued == kk + NST && i + NST - it.nb < nx_nb) {
                        // (only if every earlier position is issued: a next
                        // item learnt late takes its first stages after the loop)
                        const int j = i + NST - it.nb;  // < NST: within the first 32 entries
                        ng = nx_g;
                        npb = __shfl_sync(FULL, entn0, j);
                        nrun = nx_b0 + j;
                    }
                    __syncwarp();  // every lane's K fragments are read
                    if (ng >= 0) {
                        issue_half(0, ng, kk + NST, npb, nrun);
                        issued_k = kk + NST + 1;
                    }
                    ok = __all_sync(FULL, mbar_wait(&wbar[NST + kk % NST], (kk / NST) & 1));
                    if (!ok) break;
                    if (valid) {
                        if (nvalid < 16) path.zero_tail(vaddr, 0, nvalid, lane);
                        if constexpr (kF32)
                            path.accumulate(vaddr, 0, lane, ph, pl);
                        else if (kSpTiles<T, D> == 2 && two)
                            path.template accumulate<2>(vaddr, 0, lane, ph, pl);
                        else
                            path.template accumulate<1>(vaddr, 0, lane, ph1, pl1);
                    }
                    __syncwarp();
                    if (i == claim_at && lane == 0) jn_raw = atomicAdd(a.counter, 1);
                    if (i == read_at) {
                        jn = __shfl_sync(FULL, jn_raw, 0);
                        fn = field(jn);
                    }
                    if (i == learn_at) learn_next();
                    if (ng >= 0) {
                        issue_half(1, ng, kk + NST, npb, nrun);
                        issued = kk + NST + 1;
                    }
                    continue;
                }
                ok = __all_sync(FULL, mbar_wait(&wbar[kk % NST], (kk / NST) & 1));
                if (!ok) break;
                if (pb >= 0 && pb < a.num_blocks) {
                    const int nvalid = min(BS, it.tok_end - (it.b0 + i) * BS);
                    const uint32_t kaddr = smem_u32(wstage + (kk % NST) * Gm::kStageBytes);
                    if constexpr (kSpTiles<T, D> == 2) {
                        if (two)
                            path.template block<2, kSpRows<T, D>>(kaddr, kaddr + Gm::kTileBytes, qaddr,
                                                               nvalid, a.scale_log2, lane);
                        else
                            path.template block<1, kSpRows<T, D>>(kaddr, kaddr + Gm::kTileBytes, qaddr,
                                                               nvalid, a.scale_log2, lane);
                    } else {
                        path.template block<1, kSpRows<T, D>>(kaddr, kaddr + Gm::kTileBytes, qaddr, nvalid,
                                                           a.scale_log2, lane);
                    }
                }
                __syncwarp();
                if (i == claim_at && lane == 0) jn_raw = atomicAdd(a.counter, 1);
                if (i == read_at) {
                    jn = __shfl_sync(FULL, jn_raw, 0);
                    fn = field(jn);
                }
                if (i == learn_at) learn_next();
                if (i + NST < it.nb) {
                    issue(it.g, kk + NST, bt_get(i + NST), it.b0 + i + NST);
                    issued = kk + NST + 1;
                } else if (it.nb >= NST && i + NST - it.nb < nx_nb) {
                    // next item's block j at position ctr + nb + j, in order
                    // from j = 0 (an item shorter than NST leaves them all
                    // to after the loop)
                    const int j = i + NST - it.nb;  // < NST: within the first 32 entries
                    issue(nx_g, kk + NST, __shfl_sync(FULL, entn0, j), nx_b0 + j);
                    issued = kk + NST + 1;
                }
            }
            if (!ok) {
                if (lane == 0) raise_fault(a.dev_error, PKV_FAULT_TIMEOUT);
                // drain what this warp still has in flight, again with a bound
                if constexpr (kSplit) {
                    for (unsigned kk = ctr + i; kk < issued_k; ++kk) mbar_wait(&wbar[kk % NST], (kk / NST) & 1);
                    for (unsigned kk = ctr + i; kk < issued; ++kk) mbar_wait(&wbar[NST + kk % NST], (kk / NST) & 1);
                } else {
                    for (unsigned kk = ctr + i; kk < issued; ++kk) mbar_wait(&wbar[kk % NST], (kk / NST) & 1);
                }
                break;
            }
            if (it.nb == 0) {  // (no block ran the loop)
                jn = __shfl_sync(FULL, jn_raw, 0);
                fn = field(jn);
            }
            if (!known) learn_next();
            const bool has_next = jn < total;
            SpItem nx = it;
            if (has_next) {
                // first stages the loop did not issue (all of them when this
                // item had fewer than NST blocks), then the next query rows,
                // before this item's epilogue
                nx = decode(jn, fn);
#pragma unroll 1
                for (unsigned p = issued; p < ctr + it.nb + min(NST, nx.nb); ++p) {
                    const int j = (int)(p - ctr - it.nb);
                    issue(nx.g, p, __shfl_sync(FULL, entn0, j), nx.b0 + j);
                }
                load_rows(nx);  // every lane is past its last ldmatrix of the buffer
            }
            ctr += it.nb;
            // epilogue: rows gid and gid+8 of each tile, straight from registers
            const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
            for (int t = 0; t < kSpTiles<T, D>; ++t) {
                if (t == 1 && !two) break;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float L = path.l[t][hr];
                    L += __shfl_xor_sync(FULL, L, 1);
                    L += __shfl_xor_sync(FULL, L, 2);
                    const int r = t * 16 + gid + hr * 8;
                    const int npr = __shfl_sync(FULL, np, r);
                    if (r < it.R) {
                        const float invL = L > 0.f ? 1.f / L : 0.f;
                        const size_t sh = (size_t)(it.seq0 + r / G) * a.num_heads + it.g * G + r % G;
                        const size_t pi = sh * a.num_slots + it.slot;
                        if (npr != 1 && tig == 0)
                            a.ws_lse[pi] = L > 0.f ? path.m[t][hr] + __log2f(L) : -CUDART_INF_F;
                        if constexpr (kF32) {
                            // TF32 tiles: C elements 0 and 1 are head columns 4 apart
#pragma unroll
                            for (int g = 0; g < D / 32; ++g)
#pragma unroll
                                for (int j = 0; j < 4; ++j)
#pragma unroll
                                    for (int e = 0; e < 2; ++e) {
                                        const int d = path.col(g, j, e);
                                        const float v = path.o[g][j][2 * hr + e] * invL;
                                        if (npr == 1)
                                            store_out(a.out, sh * D + d, v, a.out_dtype);
                                        else
                                            a.ws_o[pi * D + d] = v;
                                    }
                        } else {
#pragma unroll
                            for (int n = 0; n < ND; ++n) {
                                const int d = n * 8 + 2 * tig;
                                const float2 v = make_float2(path.o[t][n][2 * hr] * invL,
                                                             path.o[t][n][2 * hr + 1] * invL);
                                if (npr == 1)
                                    store_out2(a.out, sh * D + d, v.x, v.y, a.out_dtype);
                                else
                                    *reinterpret_cast<float2 *>(a.ws_o + pi * D + d) = v;
                            }
                        }
                    }
                }
            }
            if (!has_next) break;
            it = nx;
            np = np1;
            ent0 = entn0;
            ent1 = entn1;
        }
    }
    griddep_launch();
}

template <typename T, int D, int BS>
pkv_status launch_sp_one(const SpLaunch &L) {
    auto kern = shared_prefix_decode_kernel<T, D, BS>;
    constexpr int smem = SpSmem<T, D, BS>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    static unsigned long long done_mask = 0ull;
    static int per_sm[64];
    const unsigned long long bit = 1ull << (L.device & 63);
    if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
        if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem)) != PKV_OK)
            return PKV_ERR_CUDA;
        int n = 0;
        if (cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kSpWarps * 32,
                                                                       smem)) != PKV_OK)
            return PKV_ERR_CUDA;
        __atomic_store_n(&per_sm[L.device & 63], n < 1 ? 1 : n, __ATOMIC_RELAXED);
        __atomic_fetch_or(&done_mask, bit, __ATOMIC_RELEASE);
    }
    const int grid = __atomic_load_n(&per_sm[L.device & 63], __ATOMIC_RELAXED) * sm_count(L.device);
    if (L.grid_warps) {
        *L.grid_warps = grid * kSpWarps;
        return PKV_OK;
    }
    // launched as a programmatic dependent of the planning kernel: the CTAs
    // set up while the plan finishes and wait for it in griddepcontrol.wait
    return cuda_status(
        launch_dependent(kern, dim3(grid), dim3(kSpWarps * 32), smem, L.stream, *L.tmk, *L.tmv, L.args));
}

// Every block is staged in runs of 16 rows (a 16-token block is one run).
template <typename T, int D>
pkv_status launch_sp_d(const SpLaunch &L) {
    return L.block_size == 16 ? launch_sp_one<T, D, 16>(L) : PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
