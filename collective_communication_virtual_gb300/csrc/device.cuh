// device.cuh -- element reductions and memory helpers shared by the kernels.
//
// Element semantics (the communicator-wide reading of the reductions):
//  * fp32 sum/prod: one IEEE binary32 op, round to nearest even (__fadd_rn/__fmul_rn,
//    which the compiler never contracts into an FMA);
//  * fp16/bf16 sum/prod: widen both operands to fp32 (exact), one fp32 op (RNE), round
//    to the storage type (RNE) -- every ring hop stores its partial in that type;
//  * int32 sum/prod: wrap modulo 2^32;
//  * min/max: the running partial a is kept unless the incoming b compares strictly
//    below / above it (compared as fp32 for 16-bit floats); the selected element keeps
//    its bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace vc {

// Programmatic dependent launch (Hopper and Blackwell).  A one-pass kernel first allows
// the next kernel on the stream to be scheduled, so that kernel's CTAs become resident
// while this one's last CTAs finish, then waits until the previous kernel has completed
// and its memory is visible before it touches global memory.  Both instructions do
// nothing for a launch without the attribute, so the ordering of a stream is kept.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch a one-pass kernel, with programmatic stream serialization when enabled.
template <typename... KArgs, typename... Args>
inline cudaError_t pdl_launch(void (*kernel)(KArgs...), unsigned grid, unsigned threads, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

enum { kSum = 0, kProd = 1, kMin = 2, kMax = 3 };
enum { kF32 = 0, kF16 = 1, kBF16 = 2, kI32 = 3 };

template <int DT> struct DTypeOf;
template <> struct DTypeOf<kF32> { using T = float; static constexpr int size = 4; };
template <> struct DTypeOf<kF16> { using T = __half; static constexpr int size = 2; };
template <> struct DTypeOf<kBF16> { using T = __nv_bfloat16; static constexpr int size = 2; };
template <> struct DTypeOf<kI32> { using T = int32_t; static constexpr int size = 4; };

// ---- one element, on raw bits --------------------------------------------------------

template <int OP>
__device__ __forceinline__ float op_f32(float a, float b) {
    if (OP == kSum) return __fadd_rn(a, b);
    if (OP == kProd) return __fmul_rn(a, b);
    if (OP == kMin) return (b < a) ? b : a;
    return (b > a) ? b : a;
}

template <int OP>
__device__ __forceinline__ uint32_t op_i32(uint32_t a, uint32_t b) {
    if (OP == kSum) return a + b;
    if (OP == kProd) return a * b;
    if (OP == kMin) return ((int32_t)b < (int32_t)a) ? b : a;
    return ((int32_t)b > (int32_t)a) ? b : a;
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float((uint32_t)h << 16);
}
__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) {
    return __half_as_ushort(__float2half_rn(f));
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int DT>
__device__ __forceinline__ float widen16(uint16_t h) {
    return DT == kF16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h);
}
template <int DT>
__device__ __forceinline__ uint16_t narrow16(float f) {
    return DT == kF16 ? f32_to_f16_bits(f) : f32_to_bf16_bits(f);
}

template <int DT, int OP>
__device__ __forceinline__ uint16_t op_16(uint16_t a, uint16_t b) {
    const float fa = widen16<DT>(a), fb = widen16<DT>(b);
    if (OP == kSum) return narrow16<DT>(__fadd_rn(fa, fb));
    if (OP == kProd) return narrow16<DT>(__fmul_rn(fa, fb));
    if (OP == kMin) return (fb < fa) ? b : a;
    return (fb > fa) ? b : a;
}

// One 32-bit word: one fp32/int32 element or two 16-bit elements.
//
// fp16/bf16 sum uses the packed add, which rounds the exact sum once.  That equals the
// widen / fp32 add / round definition: two 16-bit floats whose exponents differ by at
// most 13 (fp16) or 15 (bf16) have an exact sum that fits fp32's 24-bit significand, so
// the fp32 add does not round; with a larger gap the smaller operand is below half an
// ulp of the larger in the 16-bit type, and both routes return the larger operand.
// (Products are not done this way: a bf16 product in the subnormal range can round twice.)
// fp16/bf16 min and max compare both lanes at once and select bits by the lane mask.
// The packed compare is ordered, like the widened fp32 compare of the definition, and
// comparing two 16-bit floats gives the same answer as comparing their exact fp32
// values: a NaN on either side keeps the running partial a, and so does a tie (-0 / +0).
template <int DT, int OP>
__device__ __forceinline__ uint32_t op_word(uint32_t a, uint32_t b) {
    if (DT == kF32) return __float_as_uint(op_f32<OP>(__uint_as_float(a), __uint_as_float(b)));
    if (DT == kI32) return op_i32<OP>(a, b);
    if (OP == kSum && DT == kBF16) {
        const __nv_bfloat162 r = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                         *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    if (OP == kSum && DT == kF16) {
        const __half2 r = __hadd2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    if ((OP == kMin || OP == kMax) && DT == kBF16) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&b);
        const uint32_t m = OP == kMax ? __hgt2_mask(y, x) : __hlt2_mask(y, x);
        return (b & m) | (a & ~m);
    }
    if ((OP == kMin || OP == kMax) && DT == kF16) {
        const __half2 x = *reinterpret_cast<const __half2*>(&a);
        const __half2 y = *reinterpret_cast<const __half2*>(&b);
        const uint32_t m = OP == kMax ? __hgt2_mask(y, x) : __hlt2_mask(y, x);
        return (b & m) | (a & ~m);
    }
    if (OP == kProd) {
        // widen each lane, one fp32 multiply per lane, then both lanes rounded back by one
        // packed convert (round to nearest even, as narrow16 does lane by lane)
        const float lo = __fmul_rn(widen16<DT>((uint16_t)(a & 0xFFFFu)), widen16<DT>((uint16_t)(b & 0xFFFFu)));
        const float hi = __fmul_rn(widen16<DT>((uint16_t)(a >> 16)), widen16<DT>((uint16_t)(b >> 16)));
        if (DT == kBF16) {
            const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
            return *reinterpret_cast<const uint32_t*>(&r);
        }
        const __half2 r = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    const uint32_t lo = op_16<DT, OP>((uint16_t)(a & 0xFFFFu), (uint16_t)(b & 0xFFFFu));
    const uint32_t hi = op_16<DT, OP>((uint16_t)(a >> 16), (uint16_t)(b >> 16));
    return lo | (hi << 16);
}

template <int DT, int OP>
__device__ __forceinline__ uint4 op_vec(uint4 a, uint4 b) {
    return make_uint4(op_word<DT, OP>(a.x, b.x), op_word<DT, OP>(a.y, b.y),
                      op_word<DT, OP>(a.z, b.z), op_word<DT, OP>(a.w, b.w));
}

template <int DT, int OP>
__device__ __forceinline__ uint2 op_vec(uint2 a, uint2 b) {
    return make_uint2(op_word<DT, OP>(a.x, b.x), op_word<DT, OP>(a.y, b.y));
}

// Element-level op on a value held in the low bits of a u32 (scalar paths).
template <int DT, int OP>
__device__ __forceinline__ uint32_t op_elem(uint32_t a, uint32_t b) {
    if (DT == kF32 || DT == kI32) return op_word<DT, OP>(a, b);
    return op_16<DT, OP>((uint16_t)a, (uint16_t)b);
}

// ---- epilogue: out = (float)acc * scale, stored as OUT ------------------------------

template <int DT>
__device__ __forceinline__ float elem_to_f32(uint32_t v) {
    if (DT == kF32) return __uint_as_float(v);
    return widen16<DT>((uint16_t)v);
}

template <int OUT>
__device__ __forceinline__ uint32_t f32_to_elem(float f) {
    if (OUT == kF32) return __float_as_uint(f);
    return narrow16<OUT>(f);
}

// ---- memory ---------------------------------------------------------------------------

// User buffers: streamed once, so keep them out of L1.  Plain (not .nc) loads, so the
// same code is correct when a receive buffer aliases a send buffer.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 32-byte accesses (Blackwell's 256-bit global loads and stores): half the instructions
// of the 16-byte path for the same bytes in flight.  No L2 eviction hint: with the CTAs
// of a flat grid dispatched in order, plain accesses measured about 1 % faster than
// evict-first ones on GB300.
struct V32 {
    uint4 lo, hi;
};
__device__ __forceinline__ V32 ld_stream32(const void* p) {
    V32 v;
    asm("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y),
          "=r"(v.hi.z), "=r"(v.hi.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream32(void* p, const V32& v) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(v.lo.x), "r"(v.lo.y), "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x),
                    "r"(v.hi.y), "r"(v.hi.z), "r"(v.hi.w)
                 : "memory");
}
template <int DT, int OP>
__device__ __forceinline__ V32 op_vec(const V32& a, const V32& b) {
    V32 r;
    r.lo = op_vec<DT, OP>(a.lo, b.lo);
    r.hi = op_vec<DT, OP>(a.hi, b.hi);
    return r;
}

// Vector of VB bytes (16 or 32) with its load/store.
template <int VB> struct VecOf;
template <> struct VecOf<16> {
    using T = uint4;
    static __device__ __forceinline__ uint4 ld(const void* p) { return ld_stream(p); }
    static __device__ __forceinline__ void st(void* p, const uint4& v) { st_stream(p, v); }
};
template <> struct VecOf<32> {
    using T = V32;
    static __device__ __forceinline__ V32 ld(const void* p) { return ld_stream32(p); }
    static __device__ __forceinline__ void st(void* p, const V32& v) { st_stream32(p, v); }
};

// Bytes [sh, sh + 16) of the 32 bytes a, b (little endian), for sh in [0, 16).
__device__ __forceinline__ uint4 shift_bytes(const uint4& a, const uint4& b, unsigned sh) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const unsigned r = (sh & 3u) * 8u;
    uint32_t o[4];
    switch (sh >> 2) {
#define VC_SHIFT_CASE(Q)                                                                   \
    case Q:                                                                                \
        _Pragma("unroll") for (int k = 0; k < 4; k++) o[k] = __funnelshift_r(w[k + Q], w[k + Q + 1], r); \
        break;
        VC_SHIFT_CASE(0)
        VC_SHIFT_CASE(1)
        VC_SHIFT_CASE(2)
        default:
        _Pragma("unroll") for (int k = 0; k < 3; k++) o[k] = __funnelshift_r(w[k + 3], w[k + 4], r);
        o[3] = __funnelshift_r(w[6], w[7], r);
        break;
#undef VC_SHIFT_CASE
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Element loads/stores for the scalar paths (esz = 2 or 4).
template <int ESZ>
__device__ __forceinline__ uint32_t ld_elem(const void* base, size_t e) {
    if (ESZ == 4) return *((const uint32_t*)base + e);
    return *((const uint16_t*)base + e);
}
template <int ESZ>
__device__ __forceinline__ void st_elem(void* base, size_t e, uint32_t v) {
    if (ESZ == 4) *((uint32_t*)base + e) = v;
    else *((uint16_t*)base + e) = (uint16_t)v;
}

// FIFO traffic: L2 only (another SM produced it), and ordered by the protocol's flags.
__device__ __forceinline__ uint4 ld_cg(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_cg(void* p, uint4 v) {
    asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void ld_volatile_u64x2(const void* p, unsigned long long& a,
                                                  unsigned long long& b) {
    asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_volatile_u64x2(void* p, unsigned long long a,
                                                  unsigned long long b) {
    asm volatile("st.volatile.global.v2.u64 [%0], {%1,%2};" :: "l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ unsigned long long ld_volatile_u64(const void* p) {
    unsigned long long v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_volatile_u64(void* p, unsigned long long v) {
    asm volatile("st.volatile.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const void* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(void* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// First error wins (decided by an atomic on the device copy of the status word); the
// winner mirrors the record into the pinned host copy that vcommGetAsyncError reads.
__device__ __forceinline__ void report_error(Status* dev, volatile Status* host, unsigned code,
                                             unsigned ch, unsigned rank, unsigned step) {
    if (atomicCAS(&dev->code, 0u, code) == 0u) {
        dev->channel = ch;
        dev->rank = rank;
        dev->step = step;
        if (host) {
            host->channel = ch;
            host->rank = rank;
            host->step = step;
            __threadfence_system();
            host->code = code;
            __threadfence_system();
        }
    }
}

}  // namespace vc
