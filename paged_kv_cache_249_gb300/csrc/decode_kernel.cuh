// decode_kernel.cuh -- paged decode-attention kernel for sm_103a.
//
// One CTA computes the attention of the G query heads that share one KV head
// (grouped-query attention, vAttention section 3.1) of one sequence over one
// partition of its context.  The KV cache is read in place from the block
// pool through the sequence's block table (Qualiteg, "About PagedAttention
// for LLM serving", the section on logical and physical blocks), so
// every (block, kv head) tile is read from HBM once per KV head, whatever G.
//
// Data movement: each warp owns NST shared-memory stages.  Lane 0 of the warp
// stages a block's K and V tiles with 2-D TMA tiled copies (128-byte-wide
// slabs, 128-byte swizzle) that complete on the stage's mbarrier; the warp
// walks logical blocks warp, warp+NW, warp+2NW, ... of the partition.  Block
// numbers are gathered 32 at a time by the whole warp, one chunk ahead.
//
// Arithmetic (standard softmax attention, online form): scores in the log2
// domain, a running max m and sum l per query row, the accumulator rescaled
// by 2^(m_old - m_new) when the max moves.  Three compute paths:
//   * FMA: CUDA-core dot products; a row of D elements is spread over
//     LPT lanes (16-byte chunks), reduced with xor shuffles.  A CTA takes at
//     most four rows of a group; a larger group is split over CTAs.
//   * MMA: bf16 or fp16 mma.sync m16n8k16 with the G query rows padded to 16:
//     S = Q K^T per block from ldmatrix'd K, then O += P V with P split into
//     a 16-bit high part and a 16-bit remainder so the weights keep ~16 bits.
//   * TF32 (fp32 pools, larger groups): mma.sync m16n8k8 tiles, each product
//     as three TF32 products (high*high + high*low + low*high); every k-step's
//     chain starts from zero and is added to the running sum in fp32.
// The tensor-core paths keep a lazy per-row reference instead of the exact
// running max: it moves only when a score passes it by 8 (log2 units), so
// most blocks skip the rescale; the weights then stay below 2^8.
// At the end the per-warp states are merged with a log-sum-exp combine in
// shared memory; a partitioned (split) context writes normalised partials
// and their log2-sum-exp, which lse_combine reduces.
#pragma once

#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<float> {
    static constexpr int kBytes = 4;
};
template <>
struct ElemTraits<__nv_bfloat16> {
    static constexpr int kBytes = 2;
};
template <>
struct ElemTraits<__half> {
    static constexpr int kBytes = 2;
};

template <typename T, int D, int BS>
struct Geom {
    static constexpr int kElemBytes = ElemTraits<T>::kBytes;
    static constexpr int kRowBytes = D * kElemBytes;
    static constexpr int kSlabs = kRowBytes / 128;      // 128-byte-wide column slabs
    static constexpr int kSlabElems = 128 / kElemBytes;
    static constexpr int kSlabBytes = BS * 128;
    static constexpr int kTileBytes = BS * kRowBytes;   // one (block, kv head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
    static constexpr int kChunks = kRowBytes / 16;      // 16-byte chunks per row
    static constexpr int kEPC = 16 / kElemBytes;        // elements per chunk
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte slabs");
};

// Warps per CTA and the shared-memory budget of the staging ring (bytes per
// CTA); compile-time tuning knobs.
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
#ifndef PKV_STAGE_BUDGET
#define PKV_STAGE_BUDGET 65536
#endif
constexpr int kDecodeWarps = PKV_DECODE_WARPS;

template <typename T, int D, int BS>
constexpr int decode_stages() {
    constexpr int per = kDecodeWarps * Geom<T, D, BS>::kStageBytes;
    constexpr int n = PKV_STAGE_BUDGET / per;
    return n < 1 ? 1 : (n > 8 ? 8 : n);
}

// Per-warp state exported for the cross-warp merge: m[GP], l[GP], o[GP][D].
template <int GP, int D>
struct WarpState {
    float m[GP];
    float l[GP];
    float o[GP][D];
};

// Shared memory of one CTA: the staging ring, reused after the main loop for
// the warps' exported states (whichever is larger), then one mbarrier per
// stage, plus slack to align the base to 1024 bytes.
template <typename T, int D, int BS, int RG>
constexpr int decode_ring_bytes() {
    constexpr int ring = kDecodeWarps * decode_stages<T, D, BS>() * Geom<T, D, BS>::kStageBytes;
    constexpr int st = kDecodeWarps * (int)sizeof(WarpState<RG, D>);
    return ring > st ? ring : st;
}
// bytes of the TF32 path's shared query fragments (KS k-steps x 32 lanes x 16 B)
template <int D>
constexpr int tf32_qbuf_bytes() {
    return (D / 8) * 32 * 16;
}
template <typename T, int D, int BS, int RG, bool QBUF = false>
constexpr int decode_smem_bytes() {
    return decode_ring_bytes<T, D, BS, RG>() + kDecodeWarps * decode_stages<T, D, BS>() * 8 +
           (QBUF ? tf32_qbuf_bytes<D>() + 16 : 0) + 1024;
}

__device__ __forceinline__ float load_as_float(const float *p) { return *p; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ float load_as_float(const __half *p) { return __half2float(*p); }

// Load 16 bytes of q / K / V and widen to EPC floats.
template <typename T>
__device__ __forceinline__ void widen16(const uint4 &v, float *f);
template <>
__device__ __forceinline__ void widen16<float>(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void widen16<__nv_bfloat16>(const uint4 &v, float *f) {
    f[0] = bf16_lo(v.x);
    f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y);
    f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z);
    f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w);
    f[7] = bf16_hi(v.w);
}
template <>
__device__ __forceinline__ void widen16<__half>(const uint4 &v, float *f) {
    f[0] = f16_lo(v.x);
    f[1] = f16_hi(v.x);
    f[2] = f16_lo(v.y);
    f[3] = f16_hi(v.y);
    f[4] = f16_lo(v.z);
    f[5] = f16_hi(v.z);
    f[6] = f16_lo(v.w);
    f[7] = f16_hi(v.w);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ------------------------------------------------------------ FMA compute

template <typename T, int D, int BS, int GP>
struct FmaPath {
    using Gm = Geom<T, D, BS>;
    static constexpr int LPT = Gm::kChunks < 16 ? Gm::kChunks : 16;  // lanes per token
    static constexpr int CPL = Gm::kChunks / LPT;                    // chunks per lane
    static constexpr int TPP = 32 / LPT;                             // tokens per pass
    static constexpr int NI = BS / TPP;                              // passes per block
    static constexpr int EPC = Gm::kEPC;

    float q[GP][CPL][EPC];  // query rows, pre-multiplied by scale*log2(e)
    float m[GP], l[GP];
    float acc[GP][CPL][EPC];
    int tg, li;

    __device__ __forceinline__ void init(const T *qrow0, int group, float scale_log2, int lane) {
        tg = lane / LPT;
        li = lane % LPT;
#pragma unroll
        for (int r = 0; r < GP; ++r) {
            m[r] = -CUDART_INF_F;
            l[r] = 0.f;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                float f[EPC];
                if (r < group) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const char *>(qrow0 + (size_t)r * D) + (li + k * LPT) * 16);
                    widen16<T>(v, f);
                } else {
#pragma unroll
                    for (int e = 0; e < EPC; ++e) f[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    q[r][k][e] = f[e] * scale_log2;
                    acc[r][k][e] = 0.f;
                }
            }
        }
    }

    // One staged block: K tile at kaddr, V tile at vaddr (shared addresses),
    // the first `nvalid` of its BS rows are context tokens.
    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, int nvalid) {
        float sc[NI][GP];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int tok = tg + i * TPP;
            float part[GP];
#pragma unroll
            for (int r = 0; r < GP; ++r) part[r] = 0.f;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                float kf[EPC];
                widen16<T>(lds128(kaddr + swz_offset<BS>(tok, li + k * LPT)), kf);
#pragma unroll
                for (int r = 0; r < GP; ++r)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) part[r] = fmaf(q[r][k][e], kf[e], part[r]);
            }
#pragma unroll
            for (int r = 0; r < GP; ++r) {
#pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1)
                    part[r] += __shfl_xor_sync(0xffffffffu, part[r], off);
                sc[i][r] = tok < nvalid ? part[r] : -CUDART_INF_F;
            }
        }
#pragma unroll
        for (int r = 0; r < GP; ++r) {
            float mx = sc[0][r];
#pragma unroll
            for (int i = 1; i < NI; ++i) mx = fmaxf(mx, sc[i][r]);
            const float mn = fmaxf(m[r], mx);
            const float mu = mn == -CUDART_INF_F ? 0.f : mn;
            const float alpha = fast_exp2(m[r] - mu);
            m[r] = mn;
            float lsum = l[r] * alpha;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                sc[i][r] = fast_exp2(sc[i][r] - mu);
                lsum += sc[i][r];
            }
            l[r] = lsum;
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[r][k][e] *= alpha;
        }
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int tok = tg + i * TPP;
            if (tok < nvalid) {  // masked rows may hold stale bits (even NaN): never touch them
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    float vf[EPC];
                    widen16<T>(lds128(vaddr + swz_offset<BS>(tok, li + k * LPT)), vf);
#pragma unroll
                    for (int r = 0; r < GP; ++r)
#pragma unroll
                        for (int e = 0; e < EPC; ++e) acc[r][k][e] = fmaf(sc[i][r], vf[e], acc[r][k][e]);
                }
            }
        }
    }

    // Merge the TPP token streams of the warp and write the warp's state.
    __device__ __forceinline__ void finish(WarpState<GP, D> *st, int lane) {
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
            for (int r = 0; r < GP; ++r) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[r], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[r], off);
                const float mn = fmaxf(m[r], mo);
                const float mu = mn == -CUDART_INF_F ? 0.f : mn;
                const float wa = fast_exp2(m[r] - mu), wb = fast_exp2(mo - mu);
                l[r] = l[r] * wa + lo * wb;
                m[r] = mn;
#pragma unroll
                for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        const float ao = __shfl_xor_sync(0xffffffffu, acc[r][k][e], off);
                        acc[r][k][e] = acc[r][k][e] * wa + ao * wb;
                    }
            }
        }
        if (lane < LPT) {
#pragma unroll
            for (int r = 0; r < GP; ++r) {
#pragma unroll
                for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) st->o[r][(li + k * LPT) * EPC + e] = acc[r][k][e];
                if (lane == 0) {
                    st->m[r] = m[r];
                    st->l[r] = l[r];
                }
            }
        }
    }
};

// ------------------------------------------------------------ MMA compute

template <typename T, int D, int BS, int RG>
struct MmaPath {
    using MM = Mma16<T>;
    static constexpr int GP = RG;       // rows exported: 8 when the group fits rows g < 8
    static constexpr int KS = D / 16;   // k-steps of the QK^T product
    static constexpr int NT = BS / 8;   // token n-tiles per block
    static constexpr int ND = D / 8;    // head-dim n-tiles of the PV product
    static_assert(BS % 16 == 0 && D % 32 == 0, "tile shape");

    uint32_t qa[KS][4];                 // A fragments of Q (rows g, g+8)
    float o[ND][4];                     // O accumulators (rows g, g+8)
    float m0, m1, l0, l1;               // rows g and g+8: reference, lane-partial sum
    float scale_log2;
    int gid, tig;
    bool fresh;                         // no block seen yet

    __device__ __forceinline__ void init(const T *qrow0, int group, float sl2, int lane) {
        gid = lane >> 2;
        tig = lane & 3;
        scale_log2 = sl2;
        fresh = true;
        m0 = m1 = 0.f;
        l0 = l1 = 0.f;
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow0);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int c0 = (ks * 16 + 2 * tig) / 2, c1 = (ks * 16 + 8 + 2 * tig) / 2;
            qa[ks][0] = gid < group ? __ldg(q32 + (size_t)gid * (D / 2) + c0) : 0u;
            qa[ks][1] = gid + 8 < group ? __ldg(q32 + (size_t)(gid + 8) * (D / 2) + c0) : 0u;
            qa[ks][2] = gid < group ? __ldg(q32 + (size_t)gid * (D / 2) + c1) : 0u;
            qa[ks][3] = gid + 8 < group ? __ldg(q32 + (size_t)(gid + 8) * (D / 2) + c1) : 0u;
        }
#pragma unroll
        for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, int nvalid, int lane) {
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            const int row = nt * 8 + (lane & 7);
#pragma unroll
            for (int kc = 0; kc < D / 32; ++kc) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kaddr + swz_offset<BS>(row, kc * 4 + (lane >> 3)), b0, b1, b2, b3);
                MM::mma(s[nt], qa[2 * kc], b0, b1);
                MM::mma(s[nt], qa[2 * kc + 1], b2, b3);
            }
        }
        // lazy reference: m moves (and l, o are rescaled) only when a score
        // passes it by more than 8 (log2 units); weights stay at most 2^8
        if (nvalid < BS) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (nt * 8 + 2 * tig + e >= nvalid) s[nt][e] = s[nt][2 + e] = -CUDART_INF_F;
        }
        bool grow = fresh;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = fmaf(s[nt][e], scale_log2, -m0);
                s[nt][2 + e] = fmaf(s[nt][2 + e], scale_log2, -m1);
                grow |= s[nt][e] > 8.f;
                grow |= s[nt][2 + e] > 8.f;
            }
        }
        if (__any_sync(0xffffffffu, grow)) {
            float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float d0 = fresh ? mx0 : fmaxf(mx0, 0.f), d1 = fresh ? mx1 : fmaxf(mx1, 0.f);
            const float a0 = fresh ? 0.f : fast_exp2(-d0), a1 = fresh ? 0.f : fast_exp2(-d1);
            m0 += d0;
            m1 += d1;
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] -= d0;
                    s[nt][2 + e] -= d1;
                }
            fresh = false;
        }
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = fast_exp2(s[nt][e]);
                s[nt][2 + e] = fast_exp2(s[nt][2 + e]);
                ls0 += s[nt][e];
                ls1 += s[nt][2 + e];
            }
        }
        l0 += ls0;
        l1 += ls1;
#pragma unroll
        for (int kt = 0; kt < BS / 16; ++kt) {
            // P as A fragments: its 16-bit high part and the 16-bit remainder
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float *sv = s[2 * kt + j];
                ph[2 * j] = MM::pack(sv[0], sv[1]);
                ph[2 * j + 1] = MM::pack(sv[2], sv[3]);
                pl[2 * j] = MM::pack(sv[0] - MM::lo(ph[2 * j]), sv[1] - MM::hi(ph[2 * j]));
                pl[2 * j + 1] =
                    MM::pack(sv[2] - MM::lo(ph[2 * j + 1]), sv[3] - MM::hi(ph[2 * j + 1]));
            }
            const bool partial = nvalid < (kt + 1) * 16;
            const int t0 = kt * 16 + 2 * tig;
            const uint32_t mlo = (partial ? (t0 < nvalid ? 0x0000ffffu : 0u) |
                                                (t0 + 1 < nvalid ? 0xffff0000u : 0u)
                                          : 0xffffffffu);
            const uint32_t mhi = (partial ? (t0 + 8 < nvalid ? 0x0000ffffu : 0u) |
                                                (t0 + 9 < nvalid ? 0xffff0000u : 0u)
                                          : 0xffffffffu);
            const int tok = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int np = 0; np < ND / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vaddr + swz_offset<BS>(tok, np * 2 + (lane >> 4)), b0, b1, b2, b3);
                // rows past the context may hold stale bits (even NaN): zero them
                b0 &= mlo;
                b2 &= mlo;
                b1 &= mhi;
                b3 &= mhi;
                MM::mma(o[2 * np], ph, b0, b1);
                MM::mma(o[2 * np], pl, b0, b1);
                MM::mma(o[2 * np + 1], ph, b2, b3);
                MM::mma(o[2 * np + 1], pl, b2, b3);
            }
        }
    }

    __device__ __forceinline__ void finish(WarpState<GP, D> *st, int lane) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
        for (int n = 0; n < ND; ++n) {
            const int d = n * 8 + 2 * tig;
            st->o[gid][d] = o[n][0];
            st->o[gid][d + 1] = o[n][1];
            if constexpr (RG == 16) {
                st->o[gid + 8][d] = o[n][2];
                st->o[gid + 8][d + 1] = o[n][3];
            }
        }
        if (tig == 0) {
            // a warp that saw no block has no reference: it must not set M
            st->m[gid] = fresh ? -CUDART_INF_F : m0;
            st->l[gid] = l0;
            if constexpr (RG == 16) {
                st->m[gid + 8] = fresh ? -CUDART_INF_F : m1;
                st->l[gid + 8] = l1;
            }
        }
    }
};

// ------------------------------------------------------ TF32 tensor cores

// fp32 value rounded to TF32 (10-bit mantissa, nearest, ties away), as the
// 32-bit operand register of a TF32 MMA.
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// x as a TF32 high part and the TF32 rounding of its remainder
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}

// D = A(16x8 tf32, row) * B(8x8 tf32, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// a*b from three TF32 products, hi*hi + hi*lo + lo*hi (the lo*lo term is
// below 2^-22 of the product).  Callers start each chain from a zero
// accumulator and add it to their running sums with rounded fp32 adds: the
// tensor cores' own accumulation onto a large running sum loses low bits
// with a bias (on scores of ~100 in log2 units the error grew 5x above the
// CUDA-core fp32 path's; with zero-started chains it matches it)
__device__ __forceinline__ void mma_tf32x3(float (&d)[4], const uint32_t (&ah)[4],
                                           const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1,
                                           uint32_t bl0, uint32_t bl1) {
    mma_tf32_1688(d, al, bh0, bh1);
    mma_tf32_1688(d, ah, bl0, bl1);
    mma_tf32_1688(d, ah, bh0, bh1);
}


// fp32 storage on tensor cores: the G query rows (padded to 16) as m16n8k8
// TF32 tiles, each product as three TF32 products, each k-step (and each
// block's P V) from a zero accumulator added by rounded fp32 adds, so that
// scores and outputs keep about fp32 accuracy.  K fragments come from the swizzled
// stage with ldmatrix (an 8-row, 16-byte matrix of the 16-bit view holds an
// 8x4 block of fp32, one value per lane, which is what a TF32 B fragment
// wants); V fragments with 16-byte loads, four O columns at a time, so O's
// columns inside each 32-column group are permuted (column d = 32g + 4n + j
// is n-tile j's column n) and restored when the warp exports its state.
template <int D, int BS, int RG>
struct Tf32Path {
    static constexpr int KS = D / 8;   // k-steps of the QK^T product
    static constexpr int NT = BS / 8;  // token n-tiles per block (k-steps of P V)
    static constexpr int NG = D / 32;  // 32-column groups of O
    static_assert(BS == 16 && D % 32 == 0, "tile shape");

    // The query fragments sit in shared memory, one fp32 copy per CTA, and
    // are split per k-step (three TF32 parts a value would take 3 * D / 2
    // registers a thread).
    uint32_t qbuf;                  // shared fragments: [KS][lane] x 4 fp32
    float o[NG][4][4];              // O accumulators: column group, n-tile, C fragment
    float m0, m1, l0, l1;           // rows g and g+8: reference, lane-partial sum
    float scale_log2;
    int gid, tig;
    bool fresh;                     // no block seen yet

    // The CTA's warps write one copy of the fragments, each warp every
    // nwarps-th k-step, and the caller syncs the CTA before the first block.
    __device__ __forceinline__ void init(const float *qrow0, int group, float sl2, int lane,
                                         uint32_t qb, int warp, int nwarps) {
        gid = lane >> 2;
        tig = lane & 3;
        scale_log2 = sl2;
        fresh = true;
        m0 = m1 = 0.f;
        l0 = l1 = 0.f;
        qbuf = qb;
        auto qval = [&](int ks, int i) -> float {  // fragment value i of k-step ks
            const int r = gid + (i & 1) * 8, c = ks * 8 + tig + (i >> 1) * 4;
            return r < group ? __ldg(qrow0 + (size_t)r * D + c) : 0.f;
        };
        for (int ks = warp; ks < KS; ks += nwarps)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(qbuf + (ks * 32 + lane) * 16),
                         "f"(qval(ks, 0)), "f"(qval(ks, 1)), "f"(qval(ks, 2)), "f"(qval(ks, 3))
                         : "memory");
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[g][j][0] = o[g][j][1] = o[g][j][2] = o[g][j][3] = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, int nvalid, int lane) {
        // S = Q K^T: lane L names row (L & 7) of matrix L >> 3 of an ldmatrix.x4
        // whose matrices are (tokens 0-7 | 8-15) x (head columns 8ks..+3 | +4..+7)
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        const int ktok = (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint4 qv = lds128(qbuf + (ks * 32 + lane) * 16);
            const float qf[4] = {__uint_as_float(qv.x), __uint_as_float(qv.y), __uint_as_float(qv.z),
                                 __uint_as_float(qv.w)};
            uint32_t ah[4], al[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tf32_split(qf[i], ah[i], al[i]);
            uint32_t r[4];
            ldsm_x4(kaddr + swz_offset<BS>(ktok, ks * 2 + ((lane >> 3) & 1)), r[0], r[1], r[2], r[3]);
            uint32_t kh[4], kl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tf32_split(__uint_as_float(r[i]), kh[i], kl[i]);
            // each k-step from a zero accumulator, added to the scores by a
            // rounded fp32 add (the tensor cores' own accumulation, on a large
            // running sum, loses low bits with a bias)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float t[4] = {0.f, 0.f, 0.f, 0.f};
                mma_tf32x3(t, ah, al, kh[2 * nt], kh[2 * nt + 1], kl[2 * nt], kl[2 * nt + 1]);
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] += t[e];
            }
        }
        // online softmax against a lazy reference (as on the 16-bit path)
        if (nvalid < BS) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (nt * 8 + 2 * tig + e >= nvalid) s[nt][e] = s[nt][2 + e] = -CUDART_INF_F;
        }
        bool grow = fresh;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = fmaf(s[nt][e], scale_log2, -m0);
                s[nt][2 + e] = fmaf(s[nt][2 + e], scale_log2, -m1);
                grow |= s[nt][e] > 8.f;
                grow |= s[nt][2 + e] > 8.f;
            }
        if (__any_sync(0xffffffffu, grow)) {
            float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float d0 = fresh ? mx0 : fmaxf(mx0, 0.f), d1 = fresh ? mx1 : fmaxf(mx1, 0.f);
            const float a0 = fresh ? 0.f : fast_exp2(-d0), a1 = fresh ? 0.f : fast_exp2(-d1);
            m0 += d0;
            m1 += d1;
            l0 *= a0;
            l1 *= a1;
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
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] -= d0;
                    s[nt][2 + e] -= d1;
                }
            fresh = false;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[nt][e] = fast_exp2(s[nt][e]);
                (e < 2 ? l0 : l1) += s[nt][e];
            }
        // O += P V, one 8-token k-step per n-tile of S.  P moves from the C
        // layout (row g, columns 2t, 2t+1) to the A layout (row g, columns t,
        // t+4) by shuffles inside each group of four lanes.
        const int base = lane & ~3, srcA = base + (tig >> 1), srcB = srcA + 2;
        const bool odd = tig & 1;
        uint32_t ph[NT][4], pl[NT][4];
#pragma unroll
        for (int kt = 0; kt < NT; ++kt) {
            float pa[4];
            {
                const float x0 = __shfl_sync(0xffffffffu, s[kt][0], srcA);
                const float x1 = __shfl_sync(0xffffffffu, s[kt][1], srcA);
                const float y0 = __shfl_sync(0xffffffffu, s[kt][2], srcA);
                const float y1 = __shfl_sync(0xffffffffu, s[kt][3], srcA);
                const float z0 = __shfl_sync(0xffffffffu, s[kt][0], srcB);
                const float z1 = __shfl_sync(0xffffffffu, s[kt][1], srcB);
                const float w0 = __shfl_sync(0xffffffffu, s[kt][2], srcB);
                const float w1 = __shfl_sync(0xffffffffu, s[kt][3], srcB);
                pa[0] = odd ? x1 : x0;  // P[g][t]
                pa[1] = odd ? y1 : y0;  // P[g+8][t]
                pa[2] = odd ? z1 : z0;  // P[g][t+4]
                pa[3] = odd ? w1 : w0;  // P[g+8][t+4]
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) tf32_split(pa[i], ph[kt][i], pl[kt][i]);
        }
        // this block's P V from zero accumulators, added to O by rounded fp32
        // adds.  V rows past the context may hold stale bits (even NaN): they
        // are read as zero
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            float f[NT][2][4];
#pragma unroll
            for (int kt = 0; kt < NT; ++kt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = kt * 8 + tig + 4 * h;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (t < nvalid) v = lds128(vaddr + swz_offset<BS>(t, g * 8 + gid));
                    f[kt][h][0] = __uint_as_float(v.x);
                    f[kt][h][1] = __uint_as_float(v.y);
                    f[kt][h][2] = __uint_as_float(v.z);
                    f[kt][h][3] = __uint_as_float(v.w);
                }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kt = 0; kt < NT; ++kt) {
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

    __device__ __forceinline__ void finish(WarpState<RG, D> *st, int lane) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // C columns 2t and 2t+1 of n-tile j are head columns 32g + 8t + j and +4
                const int d0 = g * 32 + 8 * tig + j, d1 = d0 + 4;
                st->o[gid][d0] = o[g][j][0];
                st->o[gid][d1] = o[g][j][1];
                if constexpr (RG == 16) {
                    st->o[gid + 8][d0] = o[g][j][2];
                    st->o[gid + 8][d1] = o[g][j][3];
                }
            }
        if (tig == 0) {
            // a warp that saw no block has no reference: it must not set M
            st->m[gid] = fresh ? -CUDART_INF_F : m0;
            st->l[gid] = l0;
            if constexpr (RG == 16) {
                st->m[gid + 8] = fresh ? -CUDART_INF_F : m1;
                st->l[gid + 8] = l1;
            }
        }
    }
};

// ------------------------------------------------------------------ kernel

template <typename T, int D, int BS, int GP, bool MMA>
struct PathOf {
    using type = FmaPath<T, D, BS, GP>;
};
template <int D, int BS, int GP>
struct PathOf<__nv_bfloat16, D, BS, GP, true> {
    using type = MmaPath<__nv_bfloat16, D, BS, GP>;
};
template <int D, int BS, int GP>
struct PathOf<__half, D, BS, GP, true> {
    using type = MmaPath<__half, D, BS, GP>;
};
template <int D, int BS, int GP>
struct PathOf<float, D, BS, GP, true> {
    using type = Tf32Path<D, BS, GP>;
};

template <typename T, int D, int BS, int GP, bool MMA, bool RUNS>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
    using Gm = Geom<T, D, BS>;
    using Path = typename PathOf<T, D, BS, GP, MMA>::type;
    constexpr int NW = kDecodeWarps;
    constexpr int NST = decode_stages<T, D, BS>();
    constexpr int RG = GP;  // rows of the exported warp state
    constexpr int RING = decode_ring_bytes<T, D, BS, RG>();
    constexpr bool TF32 = MMA && sizeof(T) == 4;  // fp32 storage on tensor cores
    constexpr bool QBUF = TF32;                    // with the query fragments in shared memory

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    // kv head fastest: consecutive CTAs read neighbouring (block, kv head)
    // tiles; a group split over row_split CTAs has them side by side
    const int g = blockIdx.x / a.row_split, s = blockIdx.y, part = blockIdx.z;
    const int r0 = (blockIdx.x - g * a.row_split) * a.rows_per_cta;  // first query row of the group
    const int nrows = min(a.rows_per_cta, a.group - r0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();  // inputs written by the kernel before this one are complete

    // Gather this warp's first block numbers before the context length is
    // known (bounded by the table row), so the two dependent loads overlap.
    // (Blocks here are staged runs of BS rows: a pool block of more than BS
    // rows is 2^ushift runs, all named by its one table entry.  Only the RUNS
    // instantiations stage such blocks; the others compile the shift out.)
    const int ushift = RUNS ? a.unit_shift : 0;
    const int b0 = part * a.part_blocks;
    const int tspan = min(a.max_blocks_per_seq << ushift, b0 + a.part_blocks) - b0;
    const int nw_tbl = tspan > warp ? (tspan - warp + NW - 1) / NW : 0;
    const int32_t *bt_row = a.block_tables + (size_t)s * a.max_blocks_per_seq;
    auto bt_load = [&](int chunk) -> int {
        const int i = chunk * 32 + lane;
        if (i >= nw_tbl) return -1;
        return a.contig ? b0 + warp + i * NW : __ldg(bt_row + ((b0 + warp + i * NW) >> ushift));
    };
    int ent0 = bt_load(0), ent1 = bt_load(1);

    int ctx = __ldg(a.context_lens + s);
    if (ctx < 0 || ctx > a.ctx_cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && part == 0) raise_fault(a.dev_error, PKV_FAULT_CONTEXT);
        ctx = ctx < 0 ? 0 : a.ctx_cap;
    }
    const int nblk = (ctx + BS - 1) / BS;
    if (part > 0 && b0 >= nblk) return;  // the sequence has no such partition
    const int b1 = min(nblk, b0 + a.part_blocks);
    const int nparts = (nblk + a.part_blocks - 1) / a.part_blocks;

    unsigned char *wstage = smem + warp * NST * Gm::kStageBytes;
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + RING) + warp * NST;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NST; ++i) mbar_init(&wbar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncwarp();

    // this warp's logical blocks: b0 + warp + i*NW, i < nw (nw <= nw_tbl)
    const int span = b1 - b0;
    const int nw = span > warp ? (span - warp + NW - 1) / NW : 0;
    int cb = 0;  // chunk held in ent0
    auto bt_get = [&](int i) -> int {
        const int v0 = __shfl_sync(0xffffffffu, ent0, i & 31);
        const int v1 = __shfl_sync(0xffffffffu, ent1, i & 31);
        return (i >> 5) == cb ? v0 : v1;
    };
    const uint64_t kv_policy = l2_evict_first_policy();  // K/V tiles are read once
    auto issue = [&](int i, int pb) {
        if (lane == 0) {
            uint64_t *bar = &wbar[i % NST];
            if (pb >= 0 && pb < a.num_blocks) {
                mbar_arrive_expect_tx(bar, Gm::kStageBytes);
                unsigned char *dk = wstage + (i % NST) * Gm::kStageBytes;
                unsigned char *dv = dk + Gm::kTileBytes;
                const int run = (b0 + warp + i * NW) & ((1 << ushift) - 1);
                const int y = a.contig ? ((s * a.num_kv_heads + g) * a.num_blocks + pb) * BS
                                       : (((pb * a.num_kv_heads + g) << ushift) + run) * BS;
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

    Path path;
    const T *qrow0 = reinterpret_cast<const T *>(a.q) +
                     ((size_t)s * a.num_heads + (size_t)g * a.group + r0) * D;
    if constexpr (TF32) {
        // (the shared fragments sit after the barriers: the ring is reused
        // for the warps' states)
        constexpr int qoff = (RING + NW * NST * 8 + 15) & ~15;
        path.init(qrow0, nrows, a.scale_log2, lane, smem_u32(smem + qoff), warp, NW);
        if constexpr (QBUF) __syncthreads();  // every warp's share of the fragments is written
    } else {
        path.init(qrow0, nrows, a.scale_log2, lane);
    }

#pragma unroll 1
    for (int i = 0; i < NST && i < nw; ++i) issue(i, bt_get(i));

    int i = 0;
    bool ok = true;
#pragma unroll 1
    for (; i < nw; ++i) {
        if ((i >> 5) != cb) {
            cb = i >> 5;
            ent0 = ent1;
            ent1 = bt_load(cb + 1);
        }
        const int pb = bt_get(i);
        ok = __all_sync(0xffffffffu, mbar_wait(&wbar[i % NST], (i / NST) & 1));
        if (!ok) break;
        if (pb >= 0 && pb < a.num_blocks) {
            const int lblk = b0 + warp + i * NW;
            const int nvalid = min(BS, ctx - lblk * BS);
            const uint32_t kaddr = smem_u32(wstage + (i % NST) * Gm::kStageBytes);
            if constexpr (MMA)
                path.block(kaddr, kaddr + Gm::kTileBytes, nvalid, lane);
            else
                path.block(kaddr, kaddr + Gm::kTileBytes, nvalid);
        }
        __syncwarp();
        if (i + NST < nw) issue(i + NST, bt_get(i + NST));
    }
    if (!ok) {
        if (lane == 0) raise_fault(a.dev_error, PKV_FAULT_TIMEOUT);
        // drain what this warp still has in flight, again with a bound
        for (int j = i; j < nw && j < i + NST; ++j) mbar_wait(&wbar[j % NST], (j / NST) & 1);
    }

    // ---- merge the warps' states in the (now idle) staging ring
    __syncthreads();
    WarpState<RG, D> *states = reinterpret_cast<WarpState<RG, D> *>(smem);
    path.finish(&states[warp], lane);
    __syncthreads();

    const int G = nrows;  // this CTA's rows of the group
    const bool split = nparts > 1;
    const size_t head0 = (size_t)s * a.num_heads + (size_t)g * a.group + r0;
#pragma unroll 1
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int r = idx / D, d = idx % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            M = fmaxf(M, states[w].m[r]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const WarpState<RG, D> *ws = &states[w];
                const float f = fast_exp2(ws->m[r] - M);
                L += ws->l[r] * f;
                O += ws->o[r][d] * f;
            }
        }
        const float res = L > 0.f ? O / L : 0.f;
        if (!split) {
            const size_t oi = (head0 + r) * D + d;
            store_out(a.out, oi, res, a.out_dtype);
        } else {
            const size_t pi = (head0 + r) * a.num_parts + part;
            // the combine reads these right after the grid: keep them in L2
            const uint64_t keep = l2_evict_last_policy();
            st_f32_hint(a.ws_o + pi * D + d, res, keep);
            if (d == 0) st_f32_hint(a.ws_lse + pi, L > 0.f ? M + __log2f(L) : -CUDART_INF_F, keep);
        }
    }
    griddep_launch();
}

// Explicit-instantiation helper: launch one configuration.
template <typename T, int D, int BS, int GP, bool MMA, bool RUNS>
pkv_status launch_one(const DecodeLaunch &L) {
    auto kern = paged_decode_kernel<T, D, BS, GP, MMA, RUNS>;
    constexpr int smem = decode_smem_bytes<T, D, BS, GP, MMA && sizeof(T) == 4>();
    static_assert(smem <= 227 * 1024, "shared memory budget");
    // Raise the dynamic shared-memory limit once per device for this kernel.
    static unsigned long long done_mask = 0ull;
    const unsigned long long bit = 1ull << (L.device & 63);
    if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
        if (cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem)) != PKV_OK)
            return PKV_ERR_CUDA;
        __atomic_fetch_or(&done_mask, bit, __ATOMIC_RELEASE);
    }
    dim3 grid(L.args.num_kv_heads * L.args.row_split, L.num_seqs, L.args.num_parts);
    return cuda_status(
        launch_dependent(kern, grid, dim3(kDecodeWarps * 32), smem, L.stream, *L.tmk, *L.tmv, L.args));
}

template <typename T, int D, int BS, bool RUNS>
pkv_status launch_bs(const DecodeLaunch &L) {
    if constexpr (sizeof(T) == 2 || D <= 128) {
        if (L.mma)
            return L.group_pad <= 8 ? launch_one<T, D, BS, 8, true, RUNS>(L)
                                    : launch_one<T, D, BS, 16, true, RUNS>(L);
    }
    switch (L.group_pad) {
        case 1: return launch_one<T, D, BS, 1, false, RUNS>(L);
        case 2: return launch_one<T, D, BS, 2, false, RUNS>(L);
        case 4: return launch_one<T, D, BS, 4, false, RUNS>(L);
        default: break;
    }
    if constexpr (D <= 128) {
        // (head size 256 keeps CUDA-core rows to groups of up to 4: the
        // tensor-core path takes the larger groups)
        switch (L.group_pad) {
            case 8: return launch_one<T, D, BS, 8, false, RUNS>(L);
            case 16: return launch_one<T, D, BS, 16, false, RUNS>(L);
            default: break;
        }
    }
    return PKV_ERR_UNSUPPORTED;
}

// Every block is staged in runs of 16 rows (a 16-token block is one run).
template <typename T, int D>
pkv_status launch_d(const DecodeLaunch &L) {
    if (L.block_size != 16) return PKV_ERR_UNSUPPORTED;
    return L.runs ? launch_bs<T, D, 16, true>(L) : launch_bs<T, D, 16, false>(L);
}

}  // namespace pkv
