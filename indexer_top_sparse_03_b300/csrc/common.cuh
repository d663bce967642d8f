// Device helpers shared by the kernels of the sparse attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define SA_DEVINL __device__ __forceinline__

namespace sa {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// element loads -> fp32
// ---------------------------------------------------------------------------
SA_DEVINL float to_f32(float x) { return x; }
SA_DEVINL float to_f32(bf16 x) { return __bfloat162float(x); }
SA_DEVINL float e4m3_to_f32(uint8_t code)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
    return __half2float(__half(h));
}

// Two packed bf16 -> two fp32 (exact: bf16 is the top half of an fp32).
SA_DEVINL float2 bf16x2_to_f32x2(uint32_t v)
{
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

SA_DEVINL uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// order-preserving score keys: a > b (as floats) <=> key(a) > key(b);
// -0.0 is folded onto +0.0 so that equal scores give equal keys.
// ---------------------------------------------------------------------------
SA_DEVINL uint32_t score_key(float f)
{
    uint32_t b = (f == 0.0f) ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------------------
// legacy warp MMA (m16n8k16 bf16 -> fp32) and ldmatrix
// ---------------------------------------------------------------------------
SA_DEVINL void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same shape with K = 32 for FP8-e4m3 operands (four codes per register;
// products exact in fp32, fp32 accumulation).
SA_DEVINL void mma_16832_e4m3(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

SA_DEVINL uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SA_DEVINL void ldsm_x4(uint32_t r[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

SA_DEVINL void ldsm_x4_trans(uint32_t r[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// ---------------------------------------------------------------------------
// cp.async (16 bytes, L2 only), zero-filled when !valid
// ---------------------------------------------------------------------------
SA_DEVINL void cp_async16(void* smem, const void* gmem, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(smem_u32(smem)), "l"(gmem), "r"(n));
}
SA_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
SA_DEVINL void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N)); }

// 16-byte global load that bypasses L1 allocation (streamed data)
SA_DEVINL uint4 ldg_stream16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// L2 policy for data read exactly once (streamed caches): evicted first, so
// that data reused soon (score rows, gathered K/V) stays resident.
SA_DEVINL uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

SA_DEVINL uint4 ldg_stream16_hint(const void* p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
    return v;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor finishes;
// griddep_wait() blocks until the predecessor grid has completed and its
// memory is visible (a no-op without the attribute), griddep_launch() lets
// the successor start launching.
SA_DEVINL void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SA_DEVINL void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

SA_DEVINL float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
SA_DEVINL float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

}  // namespace sa
