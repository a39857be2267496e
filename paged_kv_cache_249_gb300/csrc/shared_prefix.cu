// shared_prefix.cu -- pkv_paged_attention_decode_shared_prefix: planning
// kernel (work list from the group description), the log-sum-exp combine of
// the per-item partials, and the host entry point.  The persistent decode
// kernel itself is in shared_prefix_kernel.cuh.
#include <math_constants.h>

#include <cmath>
#include <cstring>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Automatic part sizes.  Prefix items carry up to 32 query rows and are
// the long ones; suffix items (one sequence's own blocks, G rows) are cut
// finer so the persistent grid ends on short items.  For the prefix the
// planning kernel takes the longest of 512, 1024 and 2048 tokens that still
// gives the decode grid three prefix items for every four warps, or for
// every two warps with fp32 pools (fewer parts mean fewer partials to merge
// and fewer item starts, but with fewer items than warps the grid's warps
// are not all busy on long items and the list does not balance; the fp32
// items, bound by their TF32 arithmetic, gain less from fewer starts).  The
// workspace is sized for the shortest.
constexpr int kAutoPrefixPartition = 512;   // tokens per prefix item (automatic, shortest)
constexpr int kPlanPrefixLevels = 3;        // automatic prefix parts: 512 << 0..2 tokens
constexpr int kAutoSuffixPartition = 256;   // tokens per suffix item (automatic)
constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads <= 1024, "one class-0 range per warp: at most 32 warps");

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Partition sizes in tokens (prefix, suffix) and the partial slots a sequence
// can need: ceil(max_prefix / ptp) + ceil(max_context / pts).
struct SpSizes {
    int ptp, pts;      // tokens; -1 = one part (ptp: the shortest prefix part when automatic)
    int pp, ps;        // most prefix / suffix parts of one sequence
    int slots;
    bool auto_prefix;  // the planning kernel chooses the prefix part size
};

SpSizes sp_sizes(int partition_tokens, int max_context_len, int max_prefix_len) {
    SpSizes z;
    z.auto_prefix = partition_tokens == 0;
    const int maxp = max_prefix_len < max_context_len ? max_prefix_len : max_context_len;
    int pp, ps;
    if (partition_tokens < 0) {
        z.ptp = z.pts = -1;
        pp = maxp > 0 ? 1 : 0;
        ps = max_context_len > 0 ? 1 : 0;
    } else {
        z.ptp = partition_tokens > 0 ? partition_tokens : kAutoPrefixPartition;
        z.pts = partition_tokens > 0 ? partition_tokens : kAutoSuffixPartition;
        pp = (maxp + z.ptp - 1) / z.ptp;
        ps = (max_context_len + z.pts - 1) / z.pts;
    }
    z.pp = pp;
    z.ps = ps;
    z.slots = pp + ps > 0 ? pp + ps : 1;
    return z;
}

struct SpLayout {
    size_t header, nparts, share, entries, lse, o, total;
};

SpLayout sp_layout(int num_seqs, int num_heads, int head_dim, int slots) {
    SpLayout L;
    const size_t S = (size_t)num_seqs, rows = S * num_heads * slots;
    L.header = 0;
    L.nparts = 256;
    L.share = L.nparts + round_up(S * 4, 256);
    L.entries = L.share + round_up(S * 8, 256);
    L.lse = L.entries + round_up(S * slots * sizeof(SpEntry), 256);
    L.o = L.lse + round_up(rows * 4, 256);
    L.total = L.o + round_up(rows * head_dim * 4, 256);
    return L;
}

// ------------------------------------------------------------ planning

struct SpPlan {
    const int32_t *group_starts;
    const int32_t *prefix_lens;
    const int32_t *context_lens;
    int32_t *dev_error;
    SpEntry *entries;
    int32_t *nparts;
    int32_t *share;         // [S][2]: group leader, shared blocks
    int32_t *header;        // [0] prefix entries, [1] suffix entries, [2] work counter
    int num_groups, num_seqs;
    int ctx_cap;            // context lengths are clamped to [0, ctx_cap]
    int max_prefix_len;     // tokens (already capped by max_context_len)
    int block_size;         // tokens per pool block (a shared prefix is whole blocks)
    int pbp, pbs;           // staged runs (16 tokens) per prefix / suffix item (pbp: the
                            // shortest candidate; candidate k is pbp << k, k < pbp_levels)
    int pbp_levels;         // candidate prefix part sizes (1 when the caller fixed them)
    int target_entries;     // the longest candidate with at least this many prefix entries wins
    int pbp_shift, pbs_shift;  // log2 of pbp / pbs when a power of two, else -1
    int cls_shift_s;        // suffix size classes: (pbs - nb) >> cls_shift_s
    int members_per_item;   // floor(query rows per item / group)
    int num_heads, num_kv_heads, slots;  // recorded in the header for the run's check
    int prefix_cap;         // entries [0, prefix_cap) hold prefix items
    int suffix_cap;         // entries [prefix_cap, prefix_cap + suffix_cap) hold suffix items
};

__device__ __forceinline__ int clamp_ctx(int c, int cap) { return c < 0 ? 0 : (c > cap ? cap : c); }

// One work-list entry as two 16-byte stores: the planning kernel's stores come
// from one SM, and eight 4-byte stores to scattered entries per lane held it up
__device__ __forceinline__ void put_entry(SpEntry *dst, int4 lo, int4 hi) {
    int4 *d = reinterpret_cast<int4 *>(dst);
    d[0] = lo;
    d[1] = hi;
}

// x / d for x >= 0, with a shift when d is a power of two (sh = log2 d, else -1)
__device__ __forceinline__ int div_by(int x, int d, int sh) { return sh >= 0 ? x >> sh : x / d; }

// Items are listed largest first within each region (longest-processing-time
// order): the persistent decode grid pulls them in list order, so its last
// items are the shortest and its warps finish close together.  An item of nb
// of at most cap blocks falls in size class (cap - nb) >> shift, with shift
// the least that keeps classes below kPlanClasses (0 for cap <= 64: one class
// per size).  The order inside a class is not fixed, and nothing depends on
// it: every item writes its own partial slot.
constexpr int kPlanClasses = 64;
constexpr int kPlanSmemSeqs = 8192;

// A group as a planning warp sees it (warp-uniform).
struct PlanGroup {
    int start, end;  // members [start, end)
    int pblk;        // shared runs (0 = nothing shared)
};

// One CTA turns the group description into the work list; each warp takes
// whole groups, its lanes the group's members and items.  A group with a
// shared prefix gets ceil(members / members_per_item) x ceil(prefix blocks /
// pbp) prefix items; every sequence gets ceil(own blocks / pbs) suffix items.
// Prefix items (the largest) and suffix items go to separate regions, and the
// decode kernel takes all prefix items first.  The first pass checks each
// description and counts the items of every size class; after a scan of the
// class counts, the second pass reserves, per group, one range of entries
// for its full-size items and one entry in the right class for each ragged
// item, so a group costs a few shared-memory atomics rather than one per
// item.  Context lengths are read once, into shared memory (for up to
// kPlanSmemSeqs sequences; a larger batch reads them where they are needed).
__global__ void __launch_bounds__(kPlanThreads, 1) shared_prefix_plan_kernel(const SpPlan p) {
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int L = kPlanPrefixLevels;
    __shared__ int s_ctx[kPlanSmemSeqs];
    // items per class (prefix items once for every candidate part size), then
    // the next free entry
    __shared__ int s_clsp[L][kPlanClasses];
    __shared__ int s_clss[kPlanClasses];
    __shared__ int s_tot[2];
    // class-0 items of each warp, then its first entry (prefix: per candidate)
    __shared__ int s_w0p[L][32], s_w0s[32];
    __shared__ int s_pit[L][32];  // prefix entries of each warp's groups, per candidate
    __shared__ int s_level;       // the candidate taken
    // the decode kernel may start setting up; it waits for this grid in
    // griddepcontrol.wait before it reads anything written here
    griddep_launch();
    griddep_wait();  // inputs written by the kernel before this one are complete
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    if (tid < L * kPlanClasses) (&s_clsp[0][0])[tid] = 0;
    else if (tid < (L + 1) * kPlanClasses) s_clss[tid - L * kPlanClasses] = 0;
    const bool staged = p.num_seqs <= kPlanSmemSeqs;
    bool bad = false;
    for (int i = tid; i <= p.num_groups || i < p.num_seqs; i += blockDim.x) {
        if (i <= p.num_groups) {
            const int v = __ldg(p.group_starts + i);
            if (v < 0 || v > p.num_seqs) bad = true;
            if (i == 0 && v != 0) bad = true;
            if (i == p.num_groups && v != p.num_seqs) bad = true;
            if (i < p.num_groups && v > __ldg(p.group_starts + i + 1)) bad = true;
        }
        if (i < p.num_seqs) {
            const int c = __ldg(p.context_lens + i);
            if (c < 0 || c > p.ctx_cap) raise_fault(p.dev_error, PKV_FAULT_CONTEXT);
            if (staged) s_ctx[i] = clamp_ctx(c, p.ctx_cap);
        }
    }
    const bool flat = __syncthreads_or(bad);
    if (flat && tid == 0) raise_fault(p.dev_error, PKV_FAULT_PREFIX);
    auto ctx_of = [&](int s) -> int {
        return staged ? s_ctx[s] : clamp_ctx(__ldg(p.context_lens + s), p.ctx_cap);
    };
    const int ngr = flat ? p.num_seqs : p.num_groups;
    constexpr int BS = kMaxStageRows;  // the work list counts staged runs of 16 tokens
    const int mpi = p.members_per_item;

    // members of group gi and the runs they share; a description that breaks
    // the rules shares nothing (and is reported)
    auto group_of = [&](int gi) -> PlanGroup {
        PlanGroup G{gi, gi + 1, 0};
        if (flat) return G;
        G.start = __ldg(p.group_starts + gi);
        G.end = __ldg(p.group_starts + gi + 1);
        const int plen = __ldg(p.prefix_lens + gi);
        if (plen == 0) return G;
        bool fits = true;
        for (int s = G.start + lane; s < G.end; s += 32) fits &= plen <= ctx_of(s);
        const bool ok = __all_sync(FULL, fits) && plen > 0 && (plen & (p.block_size - 1)) == 0 &&
                        plen <= p.max_prefix_len;
        if (!ok) {
            if (lane == 0) raise_fault(p.dev_error, PKV_FAULT_PREFIX);
            return G;
        }
        if (G.end - G.start >= 2) G.pblk = plen / BS;  // one member: nothing to share
        return G;
    };
    // candidate prefix part k: pbp << k runs, its shift when a power of two,
    // and the shift that maps its item sizes onto kPlanClasses classes
    auto pb_of = [&](int k) { return p.pbp << k; };
    auto pbsh_of = [&](int k) { return p.pbp_shift >= 0 ? p.pbp_shift + k : -1; };
    auto clsh_of = [&](int k) {
        int sh = 0;
        while (((pb_of(k) - 1) >> sh) >= kPlanClasses) ++sh;
        return sh;
    };
    auto cls_s = [&](int nb) { return (p.pbs - nb) >> p.cls_shift_s; };
    // suffix items of sequence s (nq; the last one has `last` runs)
    auto suffix_of = [&](int s, int pblk, int &ctx, int &nb, int &last) -> int {
        ctx = ctx_of(s);
        nb = (ctx + BS - 1) / BS;
        const int own = nb - pblk;
        if (own <= 0) return 0;
        const int nq = div_by(own + p.pbs - 1, p.pbs, p.pbs_shift);
        last = own - (nq - 1) * p.pbs;
        return nq;
    };

    // pass 1: items per size class, the prefix items once for every candidate
    // part size.  The full-size items (class 0, most of them) are counted per
    // warp, and each warp lists its own in one range of class 0, so they take
    // no shared counter (32 warps adding to one shared-memory word queue
    // behind each other).  w0p, pit: class-0 items and entries of this warp's
    // groups per candidate; w0s: its class-0 suffix items.
    int w0p[L], pit[L], w0s = 0;
#pragma unroll
    for (int k = 0; k < L; ++k) w0p[k] = pit[k] = 0;
#pragma unroll 1
    for (int gi = warp; gi < ngr; gi += nwarps) {
        const PlanGroup G = group_of(gi);
        if (G.pblk > 0) {
            const int sets = (G.end - G.start + mpi - 1) / mpi;
#pragma unroll
            for (int k = 0; k < L; ++k) {
                if (k < p.pbp_levels) {
                    const int pb = pb_of(k);
                    const int pp = div_by(G.pblk + pb - 1, pb, pbsh_of(k));
                    const int cl = (pb - (G.pblk - (pp - 1) * pb)) >> clsh_of(k);
                    w0p[k] += sets * (pp - 1) + (cl == 0 ? sets : 0);
                    pit[k] += sets * pp;
                    if (cl != 0 && lane == k) atomicAdd(&s_clsp[k][cl], sets);
                }
            }
        }
        int full = 0;
        for (int s = G.start + lane; s < G.end; s += 32) {
            int ctx, nb, last;
            const int nq = suffix_of(s, G.pblk, ctx, nb, last);
            if (nq == 0) continue;
            const int cl = cls_s(last);
            full += nq - 1 + (cl == 0 ? 1 : 0);
            if (cl != 0) atomicAdd(&s_clss[cl], 1);
        }
        w0s += __reduce_add_sync(FULL, full);
    }
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < L; ++k) {
            s_w0p[k][warp] = w0p[k];
            s_pit[k][warp] = pit[k];
        }
        s_w0s[warp] = w0s;
    }
    __syncthreads();
    // warp r for region r: the prefix part size (warp 0: the longest candidate
    // that still gives the decode grid target_entries prefix entries; their
    // number falls as the parts grow), each warp's first class-0 entry (an
    // exclusive scan over the warps; class 0 comes first), then the exclusive
    // scan of the class counts
    if (tid < 64) {
        const int r = tid >> 5;
        int level = 0;
        if (r == 0) {
            for (int k = 1; k < p.pbp_levels; ++k) {
                const int tot = __reduce_add_sync(FULL, lane < nwarps ? s_pit[k][lane] : 0);
                if (tot >= p.target_entries) level = k;
            }
            if (lane == 0) s_level = level;
        }
        int *w0a = r == 0 ? s_w0p[level] : s_w0s;
        int *cls = r == 0 ? s_clsp[level] : s_clss;
        const int w = lane < nwarps ? w0a[lane] : 0;
        int winc = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int x = __shfl_up_sync(FULL, winc, off);
            if (lane >= off) winc += x;
        }
        w0a[lane] = winc - w;
        if (lane == 31) cls[0] = winc;
        __syncwarp();
        const int c0 = cls[2 * lane], c1 = cls[2 * lane + 1];
        int inc = c0 + c1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int x = __shfl_up_sync(FULL, inc, off);
            if (lane >= off) inc += x;
        }
        const int ex = inc - c0 - c1;
        cls[2 * lane] = ex;
        cls[2 * lane + 1] = ex + c0;
        if (lane == 31) s_tot[r] = inc;
    }
    __syncthreads();

    // pass 2: every item at a free entry of its class (class 0: the warp's range)
    const int level = s_level;
    const int pbp = pb_of(level), pbp_sh = pbsh_of(level), clsh_p = clsh_of(level);
    int c0p = s_w0p[level][warp], c0s = s_w0s[warp];
#pragma unroll 1
    for (int gi = warp; gi < ngr; gi += nwarps) {
        const PlanGroup G = group_of(gi);
        const int pp = div_by(G.pblk + pbp - 1, pbp, pbp_sh);
        if (pp > 0) {
            // item k of the group: member set k / pp, part k % pp; the full
            // parts of all sets take one range, the last parts another
            const int sets = (G.end - G.start + mpi - 1) / mpi;
            const int cl = (pbp - (G.pblk - (pp - 1) * pbp)) >> clsh_p;
            const int bf = c0p;
            c0p += sets * (pp - 1);
            int br = c0p;
            if (cl == 0) {
                c0p += sets;
            } else {
                if (lane == 0) br = atomicAdd(&s_clsp[level][cl], sets);
                br = __shfl_sync(FULL, br, 0);
            }
            for (int k = lane; k < sets * pp; k += 32) {
                const int set = k / pp, q = k - set * pp;
                const int e = q < pp - 1 ? bf + set * (pp - 1) + q : br + set;
                if (e >= p.prefix_cap) {
                    raise_fault(p.dev_error, PKV_FAULT_PREFIX);
                    continue;
                }
                const int m0 = G.start + set * mpi, b0 = q * pbp, b1 = min(G.pblk, b0 + pbp);
                put_entry(p.entries + e, make_int4(m0, min(mpi, G.end - m0), G.start, b0),
                          make_int4(b1, q, b1 * BS, 0));
            }
        }
        for (int s0 = G.start; s0 < G.end; s0 += 32) {
            const int s = s0 + lane;
            int ctx = 0, nb = 0, last = 0, nq = 0;
            if (s < G.end) nq = suffix_of(s, G.pblk, ctx, nb, last);
            // class-0 entries of these 32 members: the full items (split by an
            // exclusive scan), then the last items that are full-size too
            const int nf = nq > 0 ? nq - 1 : 0;
            int inc = nf;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x = __shfl_up_sync(FULL, inc, off);
                if (lane >= off) inc += x;
            }
            const int tot = __shfl_sync(FULL, inc, 31);
            const int base = c0s + inc - nf;
            const int cl = nq > 0 ? cls_s(last) : -1;
            const unsigned full_last = __ballot_sync(FULL, cl == 0);
            int fr = c0s + tot + __popc(full_last & ((1u << lane) - 1u));
            c0s += tot + __popc(full_last);
            if (cl > 0) fr = atomicAdd(&s_clss[cl], 1);
            for (int q = 0; q < nq; ++q) {
                const int f = q < nq - 1 ? base + q : fr;
                if (f >= p.suffix_cap) {
                    raise_fault(p.dev_error, PKV_FAULT_PREFIX);
                    continue;
                }
                const int b0 = G.pblk + q * p.pbs, b1 = min(nb, b0 + p.pbs);
                put_entry(p.entries + p.prefix_cap + f, make_int4(s, 1, s, b0), make_int4(b1, pp + q, ctx, 0));
            }
            if (s < G.end) {
                p.nparts[s] = pp + nq;
                reinterpret_cast<int2 *>(p.share)[s] = make_int2(G.start, G.pblk);
            }
        }
    }
    if (tid == 0) {
        p.header[0] = s_tot[0] < p.prefix_cap ? s_tot[0] : p.prefix_cap;
        p.header[1] = s_tot[1] < p.suffix_cap ? s_tot[1] : p.suffix_cap;
        p.header[2] = 0;  // work counter (the combine resets it after each run)
        // the geometry this plan was made for; a run checks it
        p.header[kSpHdrMagic] = kSpPlanMagic;
        p.header[kSpHdrMagic + 1] = p.num_seqs;
        p.header[kSpHdrMagic + 2] = p.num_heads;
        p.header[kSpHdrMagic + 3] = p.num_kv_heads;
        p.header[kSpHdrMagic + 4] = p.block_size;
        p.header[kSpHdrMagic + 5] = p.slots;
        p.header[kSpHdrMagic + 6] = p.prefix_cap;
        p.header[kSpHdrMagic + 7] = p.members_per_item;
    }
}

// ------------------------------------------------------------- combine

// The shared-prefix partials are stored without an L2 hint; once consumed,
// l2_discard_line drops them so they are not written back to DRAM while the
// next decode streams.

// One warp per (sequence, head): sequences with one part were written by the
// decode kernel; zero parts (empty context) give a zero row; otherwise
// out = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M), M = max_p lse_p.
// Launched as a programmatic dependent of the decode kernel.
template <int D>
__global__ void __launch_bounds__(256) shared_prefix_combine_kernel(const SpArgs a, int num_seqs) {
    constexpr int PER = D / 32;
    griddep_wait();
    if (!sp_plan_matches(a)) return;  // the decode kernel reported it
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.counter = 0;  // ready for the next run
    const int wid = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wid >= num_seqs * a.num_heads) return;
    const int s = wid / a.num_heads;
    const int np = a.nparts[s];
    if (wid % a.num_heads == 0) {
        // members must name their leader's blocks inside the shared prefix
        // (the plan records shared runs; the table has one entry per block)
        const int leader = a.seq_share[2 * s], pblk = a.seq_share[2 * s + 1] >> a.unit_shift;
        if (pblk > 0 && leader != s) {
            const int32_t *mine = a.block_tables_chk + (size_t)s * a.max_blocks_per_seq;
            const int32_t *lead = a.block_tables_chk + (size_t)leader * a.max_blocks_per_seq;
            bool bad = false;
            for (int b = lane; b < pblk; b += 32) bad |= __ldg(mine + b) != __ldg(lead + b);
            if (__any_sync(0xffffffffu, bad) && lane == 0) raise_fault(a.dev_error, PKV_FAULT_PREFIX);
        }
    }
    if (np == 1) return;
    float res[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) res[j] = 0.f;
    if (np > 1) {
        const float *lse = a.ws_lse + (size_t)wid * a.num_slots;
        const float *po = a.ws_o + (size_t)wid * a.num_slots * D + lane * PER;
        float M = -CUDART_INF_F;
        for (int q = lane; q < np; q += 32) M = fmaxf(M, lse[q]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (M != -CUDART_INF_F) {
            float den = 0.f, num[PER];
#pragma unroll
            for (int j = 0; j < PER; ++j) num[j] = 0.f;
            for (int q0 = 0; q0 < np; q0 += 32) {
                // lane q holds the weight of part q0 + q
                const float wq = q0 + lane < np ? fast_exp2(lse[q0 + lane] - M) : 0.f;
                const int nq = np - q0 < 32 ? np - q0 : 32;
#pragma unroll 4
                for (int q = 0; q < nq; ++q) {
                    const float w = __shfl_sync(0xffffffffu, wq, q);
                    den += w;
                    const float *v = po + (size_t)(q0 + q) * D;
                    if constexpr (PER == 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(v);
                        num[0] = fmaf(w, x.x, num[0]);
                        num[1] = fmaf(w, x.y, num[1]);
                        num[2] = fmaf(w, x.z, num[2]);
                        num[3] = fmaf(w, x.w, num[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < PER; ++j) num[j] = fmaf(w, v[j], num[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) res[j] = den > 0.f ? num[j] / den : 0.f;
        }
        // the partial rows are dead now: the lane at the start of each
        // 128-byte line drops it from L2
        if ((lane * PER) % 32 == 0)
            for (int q = 0; q < np; ++q) l2_discard_line(po + (size_t)q * D);
    }
    const size_t oi = (size_t)wid * D + lane * PER;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        store_out(a.out, oi + j, res[j], a.out_dtype);
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                                    int max_context_len, int max_prefix_len,
                                                    int partition_tokens) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        max_prefix_len < 0)
        return 0;
    const SpSizes z = sp_sizes(partition_tokens, max_context_len, max_prefix_len);
    return sp_layout(num_seqs, num_heads, head_dim, z.slots).total;
}

namespace pkv {
namespace {

// Host-side checks and sizes shared by the plan, the run and the combined call.
struct SpCall {
    int BS, U, unit_shift, group, dev, ctx_cap, maxp, cap_blocks;  // cap_blocks counts runs of U
    SpSizes z;
    SpLayout lay;
};

pkv_status sp_prepare(const pkv_pool *pool, int num_seqs, int num_heads, int num_kv_heads,
                      int max_blocks_per_seq, int max_context_len, int max_prefix_len,
                      int partition_tokens, void *workspace, size_t workspace_bytes, SpCall &c) {
    if (!pool || pool->magic != kPoolMagic || pool->layout != 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0 || max_prefix_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_kv_heads != pool->num_kv_heads || num_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    c.BS = pool->block_size;
    if (partition_tokens < -1 || partition_tokens > kMaxPartitionTokens ||
        (partition_tokens > 0 && partition_tokens % c.BS != 0))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    // tensor-core tiles: bf16 or fp16, or TF32 (three products each) for fp32
    // pools of head size 64 or 128
    if (pool->dtype == PKV_F32 && pool->head_dim > 128) return PKV_ERR_UNSUPPORTED;
    // blocks above kMaxStageRows tokens are staged (and listed) in runs
    c.U = c.BS < kMaxStageRows ? c.BS : kMaxStageRows;
    if (c.U != kMaxStageRows) return PKV_ERR_UNSUPPORTED;  // blocks are whole 16-row runs
    c.unit_shift = 0;
    while ((c.U << c.unit_shift) < c.BS) ++c.unit_shift;
    if (((long long)max_blocks_per_seq << c.unit_shift) >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
    c.group = num_heads / num_kv_heads;
    if (c.group > kMaxGroup) return PKV_ERR_UNSUPPORTED;
    c.z = sp_sizes(partition_tokens, max_context_len, max_prefix_len);
    c.lay = sp_layout(num_seqs, num_heads, pool->head_dim, c.z.slots);
    if (!workspace || workspace_bytes < c.lay.total) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
    if ((long long)num_seqs * c.z.slots * kMaxGroup * num_kv_heads >= (1ll << 31))
        return PKV_ERR_UNSUPPORTED;
    const long long table_cap = (long long)max_blocks_per_seq * c.BS;
    c.ctx_cap = (int)(table_cap < max_context_len ? table_cap : max_context_len);
    c.maxp = max_prefix_len < max_context_len ? max_prefix_len : max_context_len;
    c.cap_blocks = (c.ctx_cap + c.U - 1) / c.U;
    if (cuda_status(cudaGetDevice(&c.dev)) != PKV_OK) return PKV_ERR_CUDA;
    if (c.dev != pool->device) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

// The decode kernel instance for the pool's storage type and head size.
pkv_status sp_dispatch(const pkv_pool *pool, const SpLaunch &L) {
    const int hd = pool->head_dim;
    if (pool->dtype == PKV_F32)
        return hd == 64 ? launch_shared_prefix_f32_d64(L) : launch_shared_prefix_f32_d128(L);
    if (pool->dtype == PKV_F16)
        return hd == 64 ? launch_shared_prefix_f16_d64(L)
                        : (hd == 128 ? launch_shared_prefix_f16_d128(L) : launch_shared_prefix_f16_d256(L));
    return hd == 64 ? launch_shared_prefix_d64(L)
                    : (hd == 128 ? launch_shared_prefix_d128(L) : launch_shared_prefix_d256(L));
}

pkv_status sp_plan(const pkv_pool *pool, const SpCall &c, int num_seqs, int num_heads,
                   const int32_t *context_lens, const int32_t *group_starts,
                   const int32_t *prefix_lens, int num_groups, void *workspace, cudaStream_t st) {
    char *ws = static_cast<char *>(workspace);
    SpPlan p;
    std::memset(&p, 0, sizeof(p));
    p.group_starts = group_starts;
    p.prefix_lens = prefix_lens;
    p.context_lens = context_lens;
    p.dev_error = pool->dev_error;
    p.entries = reinterpret_cast<SpEntry *>(ws + c.lay.entries);
    p.nparts = reinterpret_cast<int32_t *>(ws + c.lay.nparts);
    p.share = reinterpret_cast<int32_t *>(ws + c.lay.share);
    p.header = reinterpret_cast<int32_t *>(ws + c.lay.header);
    p.num_groups = num_groups;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = pool->num_kv_heads;
    p.slots = c.z.slots;
    p.ctx_cap = c.ctx_cap;
    p.max_prefix_len = c.maxp;
    p.block_size = c.BS;
    p.pbp = c.z.ptp > 0 ? c.z.ptp / c.U
                        : ((c.maxp + c.U - 1) / c.U > 0 ? (c.maxp + c.U - 1) / c.U : 1);
    p.pbs = c.z.pts > 0 ? c.z.pts / c.U : (c.cap_blocks > 0 ? c.cap_blocks : 1);
    p.members_per_item = sp_rows_for(pool->head_dim, pool->dtype == PKV_F32 ? 4 : 2) / c.group;
    // least shift with (cap - 1) >> shift < kPlanClasses
    auto cls_shift = [](int cap) {
        int sh = 0;
        while (((cap - 1) >> sh) >= kPlanClasses) ++sh;
        return sh;
    };
    p.cls_shift_s = cls_shift(p.pbs);
    auto pow2_shift = [](int d) {
        int sh = 0;
        while ((1 << sh) < d) ++sh;
        return (1 << sh) == d ? sh : -1;
    };
    p.pbp_shift = pow2_shift(p.pbp);
    // automatic prefix parts: the kernel tries pbp << 0..kPlanPrefixLevels-1
    // and keeps three prefix items for every four warps of the decode grid
    // (every two warps for fp32 pools)
    p.pbp_levels = 1;
    p.target_entries = 0;
    if (c.z.auto_prefix) {
        int warps = 0;
        SpLaunch q;
        std::memset(&q, 0, sizeof(q));
        q.head_dim = pool->head_dim;
        q.block_size = c.U;
        q.device = c.dev;
        q.grid_warps = &warps;
        const pkv_status qs = sp_dispatch(pool, q);
        if (qs != PKV_OK) return qs;
        p.pbp_levels = kPlanPrefixLevels;
        const int per = pool->dtype == PKV_F32 ? 2 : 4;  // warps per three items
        p.target_entries = (3 * warps + per * pool->num_kv_heads - 1) / (per * pool->num_kv_heads);
    }
    p.pbs_shift = pow2_shift(p.pbs);
    p.prefix_cap = num_seqs * c.z.pp;
    p.suffix_cap = num_seqs * c.z.ps;
    return cuda_status(launch_dependent(shared_prefix_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, p));
}

pkv_status sp_run(const pkv_pool *pool, const SpCall &c, void *out, pkv_dtype out_dtype,
                  const void *query, int num_seqs, int num_heads, const int32_t *block_tables,
                  int max_blocks_per_seq, float scale, void *workspace, cudaStream_t st) {
    char *ws = static_cast<char *>(workspace);
    SpArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = query;
    a.out = out;
    a.ws_o = reinterpret_cast<float *>(ws + c.lay.o);
    a.ws_lse = reinterpret_cast<float *>(ws + c.lay.lse);
    a.block_tables = block_tables;
    a.dev_error = pool->dev_error;
    a.entries = reinterpret_cast<const SpEntry *>(ws + c.lay.entries);
    a.nparts = reinterpret_cast<const int32_t *>(ws + c.lay.nparts);
    a.seq_share = reinterpret_cast<const int32_t *>(ws + c.lay.share);
    a.block_tables_chk = block_tables;
    int32_t *header = reinterpret_cast<int32_t *>(ws + c.lay.header);
    a.counter = header + 2;
    a.count = header;
    a.suffix_base = num_seqs * c.z.pp;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.group = c.group;
    a.block_size = c.BS;
    a.unit_shift = c.unit_shift;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = pool->num_blocks;
    a.num_slots = c.z.slots;
    a.out_dtype = out_dtype;
    a.members_per_item = sp_rows_for(pool->head_dim, pool->dtype == PKV_F32 ? 4 : 2) / c.group;
    a.scale_log2 = scale * 1.4426950408889634f;

    CUtensorMap maps[2];
    std::memcpy(maps, pool->tma, sizeof(maps));
    SpLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.tmk = &maps[0];
    L.tmv = &maps[1];
    L.args = a;
    L.head_dim = pool->head_dim;
    L.block_size = c.U;
    L.stream = st;
    L.device = c.dev;
    const int hd = pool->head_dim;
    const pkv_status s1 = sp_dispatch(pool, L);
    if (s1 != PKV_OK) return s1;

    // the combine waits for the decode grid in griddepcontrol.wait, then
    // resets the work counter for the next run on the same plan
    const dim3 cgrid((unsigned)(((long long)num_seqs * num_heads + 7) / 8));
    if (hd == 64)
        return cuda_status(
            launch_dependent(shared_prefix_combine_kernel<64>, cgrid, dim3(256), 0, st, a, num_seqs));
    if (hd == 256)
        return cuda_status(
            launch_dependent(shared_prefix_combine_kernel<256>, cgrid, dim3(256), 0, st, a, num_seqs));
    return cuda_status(
        launch_dependent(shared_prefix_combine_kernel<128>, cgrid, dim3(256), 0, st, a, num_seqs));
}

bool sp_out_args_ok(void *out, pkv_dtype out_dtype, const void *query, const int32_t *block_tables,
                    float scale) {
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16 && out_dtype != PKV_F16) return false;
    if (!std::isfinite(scale)) return false;
    if (!out || !query || !block_tables) return false;
    return aligned(out, 16) && aligned(query, 16) && aligned(block_tables, 4);
}

bool sp_plan_args_ok(const int32_t *context_lens, const int32_t *group_starts,
                     const int32_t *prefix_lens, int num_groups, int num_seqs) {
    if (num_groups < 1 || num_groups > num_seqs) return false;
    if (!context_lens || !group_starts || !prefix_lens) return false;
    return aligned(context_lens, 4) && aligned(group_starts, 4) && aligned(prefix_lens, 4);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_shared_prefix_plan(const pkv_pool *pool, int num_seqs, int num_heads,
                                             int num_kv_heads, int max_blocks_per_seq,
                                             const int32_t *context_lens, int max_context_len,
                                             const int32_t *group_starts,
                                             const int32_t *prefix_lens, int num_groups,
                                             int max_prefix_len, int partition_tokens,
                                             void *workspace, size_t workspace_bytes,
                                             void *stream) {
    // host-only checks first: nothing below them touches the device
    if (pool && pool->magic == kPoolMagic && num_seqs > 0 &&
        !sp_plan_args_ok(context_lens, group_starts, prefix_lens, num_groups, num_seqs))
        return PKV_ERR_INVALID_ARG;
    SpCall c;
    const pkv_status st =
        sp_prepare(pool, num_seqs, num_heads, num_kv_heads, max_blocks_per_seq, max_context_len,
                   max_prefix_len, partition_tokens, workspace, workspace_bytes, c);
    if (st != PKV_OK || num_seqs == 0) return st;
    return sp_plan(pool, c, num_seqs, num_heads, context_lens, group_starts, prefix_lens,
                   num_groups, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" pkv_status pkv_paged_attention_decode_shared_prefix_run(
    const pkv_pool *pool, void *out, pkv_dtype out_dtype, const void *query, int num_seqs,
    int num_heads, int num_kv_heads, const int32_t *block_tables, int max_blocks_per_seq,
    int max_context_len, float scale, int max_prefix_len, int partition_tokens, void *workspace,
    size_t workspace_bytes, void *stream) {
    // host-only checks first: nothing below them touches the device
    if (pool && pool->magic == kPoolMagic && num_seqs > 0 &&
        !sp_out_args_ok(out, out_dtype, query, block_tables, scale))
        return PKV_ERR_INVALID_ARG;
    SpCall c;
    const pkv_status st =
        sp_prepare(pool, num_seqs, num_heads, num_kv_heads, max_blocks_per_seq, max_context_len,
                   max_prefix_len, partition_tokens, workspace, workspace_bytes, c);
    if (st != PKV_OK || num_seqs == 0) return st;
    return sp_run(pool, c, out, out_dtype, query, num_seqs, num_heads, block_tables,
                  max_blocks_per_seq, scale, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" pkv_status pkv_paged_attention_decode_shared_prefix(
    const pkv_pool *pool, void *out, pkv_dtype out_dtype, const void *query, int num_seqs,
    int num_heads, int num_kv_heads, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, float scale, const int32_t *group_starts,
    const int32_t *prefix_lens, int num_groups, int max_prefix_len, int partition_tokens,
    void *workspace, size_t workspace_bytes, void *stream) {
    if (pool && pool->magic == kPoolMagic && num_seqs > 0) {
        if (!sp_out_args_ok(out, out_dtype, query, block_tables, scale)) return PKV_ERR_INVALID_ARG;
        if (!sp_plan_args_ok(context_lens, group_starts, prefix_lens, num_groups, num_seqs))
            return PKV_ERR_INVALID_ARG;
    }
    SpCall c;
    const pkv_status st =
        sp_prepare(pool, num_seqs, num_heads, num_kv_heads, max_blocks_per_seq, max_context_len,
                   max_prefix_len, partition_tokens, workspace, workspace_bytes, c);
    if (st != PKV_OK || num_seqs == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const pkv_status sp = sp_plan(pool, c, num_seqs, num_heads, context_lens, group_starts,
                                  prefix_lens, num_groups, workspace, s);
    if (sp != PKV_OK) return sp;
    return sp_run(pool, c, out, out_dtype, query, num_seqs, num_heads, block_tables,
                  max_blocks_per_seq, scale, workspace, s);
}
