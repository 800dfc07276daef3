// Device-side building blocks of libtsx: hand-written inline PTX for the
// mbarrier protocol, TMA bulk tensor copies, cp.async and fences, and the
// elementwise op applied to one 16-byte vector of each operand.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "tsx_internal.h"

namespace tsx {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One lane of a fully converged warp is elected (the lowest active lane).
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The single arrival of a stage: announces the bytes its loads will deliver.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `timeout_ns` of global time.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

// ---------------------------------------------------------------- fences

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the CTA, and makes mbarrier initialisation
// visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------- TMA bulk tensor

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Ask the TMA unit to bring a box of a tensor into L2 (no shared memory, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Pull a tensor map into the TMA unit's descriptor cache ahead of its use.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Reduce-store: global[box] += shared tile, element type from the tensor map.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the n most recently committed bulk store groups have finished
// reading their shared memory.
__device__ __forceinline__ void bulk_wait_read(int n)
{
    switch (n) {
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    }
}

// All committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------ cp.async (LDGSTS)

// Copy `bytes` (16, 8 or 4) global -> shared; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src, int bytes, uint32_t src_bytes)
{
    if (bytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    else if (bytes == 8)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most n of this thread's committed groups are pending.
__device__ __forceinline__ void cp_async_wait(int n)
{
    switch (n) {
#define TSX_WAIT_CASE(k) \
    case k: asm volatile("cp.async.wait_group " #k ";" ::: "memory"); break;
        TSX_WAIT_CASE(1) TSX_WAIT_CASE(2) TSX_WAIT_CASE(3) TSX_WAIT_CASE(4) TSX_WAIT_CASE(5)
        TSX_WAIT_CASE(6) TSX_WAIT_CASE(7) TSX_WAIT_CASE(8) TSX_WAIT_CASE(9) TSX_WAIT_CASE(10)
        TSX_WAIT_CASE(11) TSX_WAIT_CASE(12) TSX_WAIT_CASE(13) TSX_WAIT_CASE(14)
#undef TSX_WAIT_CASE
    default: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    }
}

// ------------------------------------------------------------ the ops

// One fp32 element.  Explicit round-to-nearest intrinsics keep the compiler
// from contracting or reassociating; sqrt is the correctly rounded one.
template <int OP>
__device__ __forceinline__ float op_f32(float a, float b, float c)
{
    if constexpr (OP == TSX_SQRT) {
        // The square root of a negative number is NaN (IEEE 754).  Those
        // lanes are answered by selection, and the correctly rounded square
        // root is evaluated on 1 in their place, so it never meets a negative
        // operand; its out-of-range handling is left to zeros, subnormals,
        // infinities and NaN.  -0 is not negative: sqrt(-0) = -0.
        const bool neg = a < 0.f;
        const float r = __fsqrt_rn(neg ? 1.f : a);
        return neg ? __uint_as_float(0x7fffffffu) : r;
    }
    else if constexpr (OP == TSX_EXP) return expf(a);
    else if constexpr (OP == TSX_ADD) return __fadd_rn(a, b);
    else if constexpr (OP == TSX_MUL) return __fmul_rn(a, b);
    else if constexpr (OP == TSX_FMA) return __fmaf_rn(a, b, c);
    else return a;
}

__device__ __forceinline__ float u32_as_f32(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f32_as_u32(float x) { return __float_as_uint(x); }

// exp of a 16-bit element, evaluated in fp32 with CUDA's fast intrinsic
// __expf.  Its documented error is at most 2 + floor(|1.173 x|) fp32 ulps,
// i.e. a relative error below 2^-14 for every |x| <= 100, where the results
// of both 16-bit types are neither 0 nor infinite.  That is far below half
// an ulp of fp16 (2^-11 relative) and bf16 (2^-8), so after rounding to the
// element type the result is within 1 ulp of exp(x).  The elementwise
// kernels use it: measured against the form below they stream 0.6-3.8 %
// faster with it (bf16 exp [16384, 16384], 2-4 stages, GB300).
__device__ __forceinline__ float exp_for_16bit(float x) { return __expf(x); }

// exp of two 16-bit elements (widened to fp32), from the identity
// exp(x) = (2^(x log2(e) / 2))^2.  The halved argument t = RN(x * c),
// c = RN(log2(e) / 2), goes through the hardware base-2 exponential
// (ex2.approx.ftz.f32, PTX ISA) and the result is squared by an ordinary
// fp32 multiply.  Halving keeps 2^t a normal fp32 number for every result a
// 16-bit type can hold: a bf16 result is subnormal from 2^-126 down to
// 2^-133, where t >= -67; the square, which does not flush, produces the
// subnormal.  Above, t > 64 squares to infinity as exp(x) overflows.
// Error: t is within 2^-17 of x log2(e) / 2 (|t| <= 67), a relative 2^-17.5
// on 2^t and 2^-16.5 after squaring; ex2.approx adds a few fp32 ulps,
// doubled by the square, and the multiply one rounding.  In all well under
// 2^-15 relative: far below half an ulp of fp16 (2^-11) and bf16 (2^-8),
// so after rounding to the element type the result is within 1 ulp of
// exp(x).  The multiplies run on packed pairs (mul.rn.f32x2).  The row
// reduction, which is bound by instruction issue rather than by memory,
// uses it: fewer instructions per element than __expf with its subnormal
// handling (bf16 exp row sums 5321 -> 6007 GB/s, GB300).
__device__ __forceinline__ float2 exp2_for_16bit(float2 x)
{
    const float c = 0.72134752044448170368f;   // log2(e) / 2
    uint64_t v, cc, t2;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(x.x), "f"(x.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t2) : "l"(v), "l"(cc));
    float t0, t1, e0, e1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(t0), "=f"(t1) : "l"(t2));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
    uint64_t e, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(e) : "f"(e0), "f"(e1));
    asm("mul.rn.f32x2 %0, %1, %1;" : "=l"(r) : "l"(e));
    float2 out;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(out.x), "=f"(out.y) : "l"(r));
    return out;
}

// Two 16-bit elements packed in 32 bits (low half first).  fma and sqrt use
// the native 16-bit instructions (one rounding of the exact result); the
// other ops evaluate in fp32 and round once into the element type.  exp
// uses __expf, or with SQ_EXP the halving-and-squaring form.
template <int DT, int OP, bool SQ_EXP = false>
__device__ __forceinline__ uint32_t op_x2(uint32_t a, uint32_t b, uint32_t c)
{
    if constexpr (DT == TSX_F16) {
        const __half2 ha = *reinterpret_cast<const __half2*>(&a);
        __half2 r;
        if constexpr (OP == TSX_FMA) {
            // one rounding of the exact a * b + c into fp16
            r = __hfma2(ha, *reinterpret_cast<const __half2*>(&b), *reinterpret_cast<const __half2*>(&c));
        } else if constexpr (OP == TSX_SQRT) {
            r = h2sqrt(ha);   // documented round-to-nearest-even
        } else {
            const float2 fa = __half22float2(ha);
            float2 fb = make_float2(0.f, 0.f);
            if constexpr (OP == TSX_ADD || OP == TSX_MUL)
                fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
            if constexpr (OP == TSX_EXP && SQ_EXP) {
                const float2 e = exp2_for_16bit(fa);
                r = __floats2half2_rn(e.x, e.y);
            } else if constexpr (OP == TSX_EXP) {
                r = __floats2half2_rn(exp_for_16bit(fa.x), exp_for_16bit(fa.y));
            } else {
                r = __floats2half2_rn(op_f32<OP>(fa.x, fb.x, 0.f), op_f32<OP>(fa.y, fb.y, 0.f));
            }
        }
        return *reinterpret_cast<uint32_t*>(&r);
    } else {
        const __nv_bfloat162 ha = *reinterpret_cast<const __nv_bfloat162*>(&a);
        __nv_bfloat162 r;
        if constexpr (OP == TSX_FMA) {
            r = __hfma2(ha, *reinterpret_cast<const __nv_bfloat162*>(&b),
                        *reinterpret_cast<const __nv_bfloat162*>(&c));
        } else if constexpr (OP == TSX_SQRT) {
            r = h2sqrt(ha);   // documented round-to-nearest-even
        } else {
            const float2 fa = __bfloat1622float2(ha);
            float2 fb = make_float2(0.f, 0.f);
            if constexpr (OP == TSX_ADD || OP == TSX_MUL)
                fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b));
            if constexpr (OP == TSX_EXP && SQ_EXP) {
                const float2 e = exp2_for_16bit(fa);
                r = __floats2bfloat162_rn(e.x, e.y);
            } else if constexpr (OP == TSX_EXP) {
                r = __floats2bfloat162_rn(exp_for_16bit(fa.x), exp_for_16bit(fa.y));
            } else {
                r = __floats2bfloat162_rn(op_f32<OP>(fa.x, fb.x, 0.f), op_f32<OP>(fa.y, fb.y, 0.f));
            }
        }
        return *reinterpret_cast<uint32_t*>(&r);
    }
}

template <int DT, int OP, bool SQ_EXP = false>
__device__ __forceinline__ uint32_t op_word(uint32_t a, uint32_t b, uint32_t c)
{
    if constexpr (OP == TSX_COPY)
        return a;
    else if constexpr (DT == TSX_F32)
        return f32_as_u32(op_f32<OP>(u32_as_f32(a), u32_as_f32(b), u32_as_f32(c)));
    else
        return op_x2<DT, OP, SQ_EXP>(a, b, c);
}

// The op on one 16-byte vector of each operand: 4 fp32 or 8 16-bit elements.
template <int DT, int OP, bool SQ_EXP = false>
__device__ __forceinline__ uint4 op_vec16(const uint4& a, const uint4& b, const uint4& c)
{
    uint4 r;
    r.x = op_word<DT, OP, SQ_EXP>(a.x, b.x, c.x);
    r.y = op_word<DT, OP, SQ_EXP>(a.y, b.y, c.y);
    r.z = op_word<DT, OP, SQ_EXP>(a.z, b.z, c.z);
    r.w = op_word<DT, OP, SQ_EXP>(a.w, b.w, c.w);
    return r;
}

}  // namespace dev
}  // namespace tsx
