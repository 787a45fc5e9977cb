// device_common.cuh -- inline-PTX building blocks shared by the sm_103a kernels:
// mbarriers with time-bounded waits, TMA (cp.async.bulk.tensor) loads/stores,
// ldmatrix / movmatrix / mma.sync fragments, bf16 packing and exp2.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernel_params.h"

namespace apex {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Record the first problem code in the per-device status word.
__device__ __forceinline__ void report_status(uint32_t *status, uint32_t code)
{
    if (status) atomicCAS(status, 0u, code);
}

// Wait until the phase with parity `parity` of the barrier has completed, for
// at most `timeout_ns` nanoseconds.  On time-out the status word is set and
// the caller goes on as if the wait had succeeded, so that every thread still
// reaches every later barrier and the kernel ends (with unspecified output).
// The global timer is read only once every 256 polls: reading it is slow, and
// polling it on every iteration delays the wake-up after the phase completes.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &wc)
{
    if (mbar_try_wait(bar, parity)) return;
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return;
        if ((n & 255u) == 0) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > wc.timeout_ns) {
                report_status(wc.status, kStatusWaitTimeout);
                return;
            }
        }
    }
}

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int x, int y,
                                            int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
        "%5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 4-D tiled store shared -> global, tracked by the issuing thread's bulk groups;
// elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// The thread's committed bulk stores have completed (writes performed).
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16, bf16, row) * B(16x8, bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- numerics
// Pack two floats to bf16x2 (round to nearest even): lo -> bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Rotate the interleaved pair held in one bf16x2 word by (c, s):
// (x0, x1) -> (x0 c - x1 s, x0 s + x1 c), computed in fp32, rounded to bf16.
__device__ __forceinline__ uint32_t rope_pair_bf16(uint32_t w, float c, float s)
{
    const float x0 = bf16lo_to_f32(w), x1 = bf16hi_to_f32(w);
    const float y0 = fmaf(x0, c, -x1 * s);
    const float y1 = fmaf(x0, s, x1 * c);
    return pack_bf16x2(y0, y1);
}

// ---- packed fp32 pairs (f32x2): one 64-bit register holds (lo, hi)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_neg(uint64_t a) { return a ^ 0x8000000080000000ull; }

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Launch a prefill kernel as a programmatic dependent of the stream's previous
// work (its blocks wait in griddepcontrol.wait before touching global memory).
template <typename K, typename... A>
inline cudaError_t launch_dependent(K kernel, int grid, int threads, int smem, cudaStream_t stream, const A &...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Sets to -inf the scores of a 128-key row that lie outside the row's visible
// keys [lo, hi] (tile-relative). Where every row of the warp has one bound off
// the tile (the causal diagonal: lo <= 0; the window's far edge: hi >= 127), a
// single comparison per key does; branch-free inside each case.
__device__ __forceinline__ void mask_row128(uint32_t (&v)[128], int lo, int hi)
{
    const uint32_t ninf = 0xff800000u;
    if (__all_sync(0xffffffffu, lo <= 0)) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
            if (e > hi) v[e] = ninf;
    } else if (__all_sync(0xffffffffu, hi >= 127)) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
            if (e < lo) v[e] = ninf;
    } else {
#pragma unroll
        for (int e = 0; e < 128; ++e)
            if (e < lo || e > hi) v[e] = ninf;
    }
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile that a
// TMA load wrote with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, tile base
// 1024-byte aligned): the chunk index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk)
{
    return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}

}  // namespace apex
