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
// mma.sync tiles), while "suffix items" walk each sequence's own blocks.
// Every item leaves a normalised partial output and its log2-sum-exp per
// query row; the combine pass merges them, which is exact for softmax.
//
// Work is a list written by a planning kernel and pulled by a persistent grid
// (one atomic counter), prefix items first, so CTAs stay busy to the end and
// no CTA is launched for an empty partition.
#pragma once

#include <math_constants.h>

#include "decode_kernel.cuh"

namespace pkv {

constexpr int kSpWarps = 4;
#ifndef PKV_SP_STAGE_BUDGET
#define PKV_SP_STAGE_BUDGET 98304
#endif

template <int D, int BS>
constexpr int sp_stages() {
    constexpr int per = kSpWarps * Geom<__nv_bfloat16, D, BS>::kStageBytes;
    constexpr int n = PKV_SP_STAGE_BUDGET / per;
    return n < 2 ? 2 : (n > 8 ? 8 : n);
}

// Per-warp state exported for the cross-warp merge.
template <int D>
struct SpState {
    float m[kSpRowsMax];
    float l[kSpRowsMax];
    float o[kSpRowsMax][D];
};

// Shared memory: [ring | warp states] (aliased: the states are written only
// once the ring is idle), the query tile, the mbarriers, the item header.
template <int D, int BS>
struct SpSmem {
    static constexpr int kRing = kSpWarps * sp_stages<D, BS>() * Geom<__nv_bfloat16, D, BS>::kStageBytes;
    static constexpr int kStates = kSpWarps * (int)sizeof(SpState<D>);
    static constexpr int kRegion = ((kRing > kStates ? kRing : kStates) + 1023) / 1024 * 1024;
    static constexpr int kQ = kSpRowsMax * D * 2;  // bf16 rows, 128-byte slabs, swizzled
    static constexpr int kBars = kSpWarps * sp_stages<D, BS>() * 8;
    static constexpr int kMisc = 256;
    static constexpr int kBytes = kRegion + kQ + kBars + kMisc + 1024;
};

// ------------------------------------------------------ tensor-core rows

// Online-softmax attention of up to two 16-row tiles of query rows against
// 16-token sub-blocks of K and V staged in shared memory.  The query tile is
// read from shared memory with ldmatrix (it would not fit in registers next
// to two tiles of accumulators); P is split into a bf16 high part and a bf16
// remainder so the weights keep about 16 bits.
template <int D, int BS>
struct SpMma {
    static constexpr int ND = D / 8;  // n-tiles of O
    float o[2][ND][4];
    float m[2][2], l[2][2];  // [tile][row gid / gid+8]; l is lane-partial
    int gid, tig;

    __device__ __forceinline__ void reset(int lane) {
        gid = lane >> 2;
        tig = lane & 3;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            m[t][0] = m[t][1] = -CUDART_INF_F;
            l[t][0] = l[t][1] = 0.f;
#pragma unroll
            for (int n = 0; n < ND; ++n) o[t][n][0] = o[t][n][1] = o[t][n][2] = o[t][n][3] = 0.f;
        }
    }

    // Tokens r0 .. r0+15 of the staged block (K at kaddr, V at vaddr), the
    // first `nvalid` (1..16) of which are context tokens; query tile at qaddr.
    template <int MT>
    __device__ __forceinline__ void sub_block(uint32_t kaddr, uint32_t vaddr, uint32_t qaddr,
                                              int r0, int nvalid, float scale_log2, int lane) {
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
                    ldsm_x4(qaddr + swz_offset<kSpRowsMax>(qrow, (2 * kc + h) * 2 + (lane >> 4)),
                            qa[t][h][0], qa[t][h][1], qa[t][h][2], qa[t][h][3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kaddr + swz_offset<BS>(r0 + nt * 8 + (lane & 7), kc * 4 + (lane >> 3)), b0,
                        b1, b2, b3);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    mma_bf16_16816(s[t][nt], qa[t][0], b0, b1);
                    mma_bf16_16816(s[t][nt], qa[t][1], b2, b3);
                }
            }
        }
        // online softmax per row (log2 domain)
        uint32_t ph[MT][4], pl[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool ok = nt * 8 + 2 * tig + e < nvalid;
                    s[t][nt][e] = ok ? s[t][nt][e] * scale_log2 : -CUDART_INF_F;
                    s[t][nt][2 + e] = ok ? s[t][nt][2 + e] * scale_log2 : -CUDART_INF_F;
                    mx0 = fmaxf(mx0, s[t][nt][e]);
                    mx1 = fmaxf(mx1, s[t][nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
            const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
            const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
            const float a0 = fast_exp2(m[t][0] - mu0), a1 = fast_exp2(m[t][1] - mu1);
            m[t][0] = mn0;
            m[t][1] = mn1;
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[t][nt][e] = fast_exp2(s[t][nt][e] - mu0);
                    s[t][nt][2 + e] = fast_exp2(s[t][nt][2 + e] - mu1);
                    ls0 += s[t][nt][e];
                    ls1 += s[t][nt][2 + e];
                }
            l[t][0] = l[t][0] * a0 + ls0;
            l[t][1] = l[t][1] * a1 + ls1;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                o[t][n][0] *= a0;
                o[t][n][1] *= a0;
                o[t][n][2] *= a1;
                o[t][n][3] *= a1;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float *sv = s[t][j];
                ph[t][2 * j] = pack_bf16(sv[0], sv[1]);
                ph[t][2 * j + 1] = pack_bf16(sv[2], sv[3]);
                pl[t][2 * j] = pack_bf16(sv[0] - bf16_lo(ph[t][2 * j]), sv[1] - bf16_hi(ph[t][2 * j]));
                pl[t][2 * j + 1] =
                    pack_bf16(sv[2] - bf16_lo(ph[t][2 * j + 1]), sv[3] - bf16_hi(ph[t][2 * j + 1]));
            }
        }
        // O += P V; rows past the context may hold stale bits (even NaN): zero them
        const bool partial = nvalid < 16;
        const int t0 = 2 * tig;
        const uint32_t mlo = partial ? ((t0 < nvalid ? 0x0000ffffu : 0u) |
                                        (t0 + 1 < nvalid ? 0xffff0000u : 0u))
                                     : 0xffffffffu;
        const uint32_t mhi = partial ? ((t0 + 8 < nvalid ? 0x0000ffffu : 0u) |
                                        (t0 + 9 < nvalid ? 0xffff0000u : 0u))
                                     : 0xffffffffu;
        const int tok = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int np = 0; np < ND / 2; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vaddr + swz_offset<BS>(tok, np * 2 + (lane >> 4)), b0, b1, b2, b3);
            b0 &= mlo;
            b2 &= mlo;
            b1 &= mhi;
            b3 &= mhi;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                mma_bf16_16816(o[t][2 * np], ph[t], b0, b1);
                mma_bf16_16816(o[t][2 * np], pl[t], b0, b1);
                mma_bf16_16816(o[t][2 * np + 1], ph[t], b2, b3);
                mma_bf16_16816(o[t][2 * np + 1], pl[t], b2, b3);
            }
        }
    }

    template <int MT>
    __device__ __forceinline__ void block(uint32_t kaddr, uint32_t vaddr, uint32_t qaddr, int nvalid,
                                          float scale_log2, int lane) {
#pragma unroll
        for (int h = 0; h < BS / 16; ++h) {
            const int nv = nvalid - h * 16;
            if (nv > 0) sub_block<MT>(kaddr, vaddr, qaddr, h * 16, nv < 16 ? nv : 16, scale_log2, lane);
        }
    }

    template <int MT>
    __device__ __forceinline__ void finish(SpState<D> *st) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float l0 = l[t][0], l1 = l[t][1];
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            const int r = t * 16 + gid;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                const int d = n * 8 + 2 * tig;
                *reinterpret_cast<float2 *>(&st->o[r][d]) = make_float2(o[t][n][0], o[t][n][1]);
                *reinterpret_cast<float2 *>(&st->o[r + 8][d]) = make_float2(o[t][n][2], o[t][n][3]);
            }
            if (tig == 0) {
                st->m[r] = m[t][0];
                st->l[r] = l0;
                st->m[r + 8] = m[t][1];
                st->l[r + 8] = l1;
            }
        }
    }
};

// ------------------------------------------------------------------ kernel

template <int D, int BS>
__global__ void __launch_bounds__(kSpWarps * 32)
    shared_prefix_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv, const SpArgs a) {
    using Gm = Geom<__nv_bfloat16, D, BS>;
    using Sm = SpSmem<D, BS>;
    constexpr int NW = kSpWarps;
    constexpr int NST = sp_stages<D, BS>();
    constexpr int QCH = D * 2 / 16;  // 16-byte chunks per query row

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *qtile = smem + Sm::kRegion;
    uint64_t *bars = reinterpret_cast<uint64_t *>(qtile + Sm::kQ);
    int *misc = reinterpret_cast<int *>(reinterpret_cast<unsigned char *>(bars) + Sm::kBars);
    int *s_next = misc;          // next item index
    int *s_np = misc + 32;       // partial count of each row's sequence
    SpState<D> *states = reinterpret_cast<SpState<D> *>(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.num_kv_heads, G = a.group;
    unsigned char *wstage = smem + warp * NST * Gm::kStageBytes;
    uint64_t *wbar = bars + warp * NST;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NST; ++i) mbar_init(&wbar[i], 1);
        fence_mbar_init();
        if (warp == 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
    }
    if (threadIdx.x == 0) *s_next = atomicAdd(a.counter, 1);
    __syncthreads();
    const int total = __ldg(a.count) * Hkv;

    SpMma<D, BS> path;
    unsigned ctr = 0;  // blocks this warp has consumed (stage ring position, across items)
    bool alive = true;
#pragma unroll 1
    for (;;) {
        const int item = *s_next;
        if (item >= total) break;
        __syncthreads();  // every thread has read s_next; the previous item's merge is done
        if (threadIdx.x == 0) *s_next = atomicAdd(a.counter, 1);
        const int e = item / Hkv, g = item - e * Hkv;
        const SpEntry en = a.entries[e];
        const int R = en.nseq * G;
        const bool two = R > 16;
        const int32_t *bt_row = a.block_tables + (size_t)en.tbl_seq * a.max_blocks_per_seq;

        // this warp's logical blocks: en.b0 + warp + i*NW, i < nw
        const int span = en.b1 - en.b0;
        const int nw = span > warp ? (span - warp + NW - 1) / NW : 0;
        auto bt_load = [&](int chunk) -> int {
            const int i = chunk * 32 + lane;
            if (i >= nw) return -1;
            const int blk = en.b0 + warp + i * NW;
            const int pb = __ldg(bt_row + blk);
            if (en.check) {  // members must name the same physical block
                bool bad = false;
                for (int m = 0; m < en.nseq; ++m) {
                    const int sq = en.seq0 + m;
                    if (sq != en.tbl_seq &&
                        __ldg(a.block_tables + (size_t)sq * a.max_blocks_per_seq + blk) != pb)
                        bad = true;
                }
                if (bad) raise_fault(a.dev_error, PKV_FAULT_PREFIX);
            }
            return pb;
        };
        int ent0 = bt_load(0), ent1 = bt_load(1);
        int cb = 0;
        auto bt_get = [&](int i) -> int {
            const int v0 = __shfl_sync(0xffffffffu, ent0, i & 31);
            const int v1 = __shfl_sync(0xffffffffu, ent1, i & 31);
            return (i >> 5) == cb ? v0 : v1;
        };
        auto issue = [&](int i, int pb) {
            if (lane == 0) {
                const unsigned k = ctr + i;
                uint64_t *bar = &wbar[k % NST];
                if (pb >= 0 && pb < a.num_blocks) {
                    mbar_arrive_expect_tx(bar, Gm::kStageBytes);
                    unsigned char *dk = wstage + (k % NST) * Gm::kStageBytes;
                    unsigned char *dv = dk + Gm::kTileBytes;
                    const int y = (pb * Hkv + g) * BS;
#pragma unroll
                    for (int sl = 0; sl < Gm::kSlabs; ++sl) {
                        tma_load_2d(dk + sl * Gm::kSlabBytes, &tmk, sl * Gm::kSlabElems, y, bar);
                        tma_load_2d(dv + sl * Gm::kSlabBytes, &tmv, sl * Gm::kSlabElems, y, bar);
                    }
                } else {
                    raise_fault(a.dev_error, PKV_FAULT_BLOCK_ID);
                    mbar_arrive(bar);
                }
            }
        };
#pragma unroll 1
        for (int i = 0; i < NST && i < nw; ++i) issue(i, bt_get(i));

        // query rows of the item (zero rows pad the last 16-row tile)
        const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
        const int rows_pad = two ? 32 : 16;
#pragma unroll 1
        for (int idx = threadIdx.x; idx < rows_pad * QCH; idx += NW * 32) {
            const int r = idx / QCH, c = idx - r * QCH;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < R) {
                const int sq = en.seq0 + r / G, h = g * G + r % G;
                v = __ldg(reinterpret_cast<const uint4 *>(q + ((size_t)sq * a.num_heads + h) * D) + c);
            }
            *reinterpret_cast<uint4 *>(qtile + swz_offset<kSpRowsMax>(r, c)) = v;
        }
        if (threadIdx.x < R) s_np[threadIdx.x] = __ldg(a.nparts + en.seq0 + threadIdx.x / G);
        __syncthreads();

        path.reset(lane);
        const uint32_t qaddr = smem_u32(qtile);
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
            const unsigned k = ctr + i;
            ok = __all_sync(0xffffffffu, mbar_wait(&wbar[k % NST], (k / NST) & 1));
            if (!ok) break;
            if (pb >= 0 && pb < a.num_blocks) {
                const int lblk = en.b0 + warp + i * NW;
                const int nvalid = min(BS, en.tok_end - lblk * BS);
                const uint32_t kaddr = smem_u32(wstage + (k % NST) * Gm::kStageBytes);
                if (two)
                    path.template block<2>(kaddr, kaddr + Gm::kTileBytes, qaddr, nvalid, a.scale_log2, lane);
                else
                    path.template block<1>(kaddr, kaddr + Gm::kTileBytes, qaddr, nvalid, a.scale_log2, lane);
            }
            __syncwarp();
            if (i + NST < nw) issue(i + NST, bt_get(i + NST));
        }
        if (!ok) {
            if (lane == 0) raise_fault(a.dev_error, PKV_FAULT_TIMEOUT);
            // drain what this warp still has in flight, again with a bound
            for (int j = i; j < nw && j < i + NST; ++j) {
                const unsigned k = ctr + j;
                mbar_wait(&wbar[k % NST], (k / NST) & 1);
            }
            alive = false;
        }
        ctr += nw;

        // ---- merge the warps' states in the (now idle) ring
        __syncthreads();
        if (two)
            path.template finish<2>(&states[warp]);
        else
            path.template finish<1>(&states[warp]);
        __syncthreads();
#pragma unroll 1
        for (int idx = threadIdx.x; idx < R * D; idx += NW * 32) {
            const int r = idx / D, d = idx - r * D;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, states[w].m[r]);
            float L = 0.f, O = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float f = fast_exp2(states[w].m[r] - M);
                    L += states[w].l[r] * f;
                    O += states[w].o[r][d] * f;
                }
            }
            const float res = L > 0.f ? O / L : 0.f;
            const int sq = en.seq0 + r / G, h = g * G + r % G;
            const size_t sh = (size_t)sq * a.num_heads + h;
            if (s_np[r] == 1) {
                if (a.out_bf16)
                    reinterpret_cast<__nv_bfloat16 *>(a.out)[sh * D + d] = __float2bfloat16_rn(res);
                else
                    reinterpret_cast<float *>(a.out)[sh * D + d] = res;
            } else {
                const size_t pi = sh * a.num_slots + en.slot;
                a.ws_o[pi * D + d] = res;
                if (d == 0) a.ws_lse[pi] = L > 0.f ? M + __log2f(L) : -CUDART_INF_F;
            }
        }
        // the next item's TMA copies overwrite the states: order this thread's
        // generic shared-memory accesses before them
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // a warp that gave up leaves the CTA's loop once the merge is done
        if (__syncthreads_or(!alive)) break;
    }
}

template <int D, int BS>
pkv_status launch_sp_one(const SpLaunch &L) {
    auto kern = shared_prefix_decode_kernel<D, BS>;
    constexpr int smem = SpSmem<D, BS>::kBytes;
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
    kern<<<grid, kSpWarps * 32, smem, L.stream>>>(*L.tmk, *L.tmv, L.args);
    return cuda_status(cudaGetLastError());
}

template <int D>
pkv_status launch_sp_d(const SpLaunch &L) {
    switch (L.block_size) {
        case 16: return launch_sp_one<D, 16>(L);
        case 32: return launch_sp_one<D, 32>(L);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace pkv
