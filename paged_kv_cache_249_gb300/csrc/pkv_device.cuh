// pkv_device.cuh -- device-side building blocks for sm_103a: mbarrier waits
// with a time bound, TMA tiled loads, ldmatrix / mma.sync wrappers, bf16 and
// fp16 packing and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// Upper bound on a single pipeline wait before the kernel gives up, records
// PKV_FAULT_TIMEOUT and stops issuing work (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void raise_fault(int32_t *err, unsigned bits) {
    if (err) atomicOr(reinterpret_cast<unsigned *>(err), bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------- programmatic dependent launch

// Wait until the grid this one was launched behind (as a programmatic
// dependent) has completed and its writes are visible; a no-op otherwise.
// Every read of a kernel input comes after it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid in the stream, if launched as a programmatic dependent,
// start its set-up now (it still waits in griddep_wait for this grid to end).
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` as a programmatic dependent of the previous kernel in
// `stream`: its CTAs may be scheduled while that kernel finishes.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Wait for `phase` of `bar` to complete.  Returns false if the wait ran past
// limit_ns (the caller then records PKV_FAULT_TIMEOUT and stops).
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, unsigned phase,
                                              unsigned long long limit_ns) {
    if (mbar_try_wait(bar, phase)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, phase)) return true;
        if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned phase) {
    return mbar_wait_for(bar, phase, kWaitLimitNs);
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box at element coordinates (x, y) into shared memory,
// completing `bar`'s transaction count.  x must be a multiple of 16 bytes /
// element size (TMA alignment rule); callers pass slab starts (128-byte steps).
// L2 policy for data read once (K/V tiles): evict first, so that what is
// read again soon (split partials, queries, tables) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data read again soon (split partials): evict last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Drop one 128-byte line of dead scratch (a partial already consumed) from L2
// without writing it back; its contents become undefined.  Split partials
// are written and read back through L2; a consumed line that stays dirty
// there is written back to DRAM while the next decode streams.
__device__ __forceinline__ void l2_discard_line(const void *p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Stores with an L2 cache policy.
__device__ __forceinline__ void st_f32_hint(float *ptr, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(policy)
                 : "memory");
}

// The same tiled load with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, int x,
                                                 int y, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar))
        : "memory");
}

// Byte offset of 16-byte chunk `c` of row `r` inside a tile staged as
// 128-byte-wide slabs with the 128-byte TMA swizzle: slab c/8, chunk c%8 of
// the slab XOR-ed with the row's position in its 8-row group.
template <int ROWS>
__device__ __forceinline__ uint32_t swz_offset(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (ROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Zero one 16-byte chunk of shared memory.
__device__ __forceinline__ void sts_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy accesses (a TMA refill of the same slot).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ tensor cores

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x16 fp16, row) * B(16x8 fp16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ numbers

// 2^x with the hardware approximation (ex2.approx, about 2 ulp); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 in one 32-bit word -> the floats they denote (bf16 is the upper
// half of an IEEE binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two fp16 in one 32-bit word -> the floats they denote, and back.
__device__ __forceinline__ float f16_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The 16-bit element types the tensor-core paths take: the mma.sync of that
// type (A and B of one type) and the packing of P into its A fragments.
template <typename T>
struct Mma16;
template <>
struct Mma16<__nv_bfloat16> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        mma_bf16_16816(d, a, b0, b1);
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16(lo, hi); }
    static __device__ __forceinline__ float lo(uint32_t w) { return bf16_lo(w); }
    static __device__ __forceinline__ float hi(uint32_t w) { return bf16_hi(w); }
};
template <>
struct Mma16<__half> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        mma_f16_16816(d, a, b0, b1);
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16(lo, hi); }
    static __device__ __forceinline__ float lo(uint32_t w) { return f16_lo(w); }
    static __device__ __forceinline__ float hi(uint32_t w) { return f16_hi(w); }
};

// Store one output value in the caller's output type (a pkv_dtype).
__device__ __forceinline__ void store_out(void *out, size_t i, float v, int out_dtype) {
    if (out_dtype == PKV_BF16)
        reinterpret_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
    else if (out_dtype == PKV_F16)
        reinterpret_cast<__half *>(out)[i] = __float2half_rn(v);
    else
        reinterpret_cast<float *>(out)[i] = v;
}
// Two adjacent output values (i even).
__device__ __forceinline__ void store_out2(void *out, size_t i, float v0, float v1, int out_dtype) {
    if (out_dtype == PKV_BF16)
        *reinterpret_cast<uint32_t *>(reinterpret_cast<__nv_bfloat16 *>(out) + i) = pack_bf16(v0, v1);
    else if (out_dtype == PKV_F16)
        *reinterpret_cast<uint32_t *>(reinterpret_cast<__half *>(out) + i) = pack_f16(v0, v1);
    else
        *reinterpret_cast<float2 *>(reinterpret_cast<float *>(out) + i) = make_float2(v0, v1);
}

}  // namespace pkv
