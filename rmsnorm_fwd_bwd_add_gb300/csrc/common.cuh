// common.cuh -- device helpers shared by the RMSNorm kernels (sm_103a).
//
// 16-byte vectors of eight fp16/bf16 values (or four fp32), fp32 conversion
// with round-to-nearest-even, warp sums in a fixed order, and inline-PTX wrappers
// for mbarriers and the 1-D TMA bulk copy (cp.async.bulk) that stages rows
// into shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace rmsn {

// Kernel modes.  MODE_VJP_ADD is the VJP of the two-output fused op: the
// plain VJP plus the gradient that reaches new_residual (a third input).
enum : int { MODE_FWD_RES = 0, MODE_FWD_NORES = 1, MODE_VJP = 2, MODE_VJP_ADD = 3 };

__host__ __device__ constexpr bool is_vjp(int mode) { return mode == MODE_VJP || mode == MODE_VJP_ADD; }
__host__ __device__ constexpr int input_tensors(int mode) {
    return mode == MODE_FWD_NORES ? 1 : mode == MODE_VJP_ADD ? 3 : 2;
}

// Bits of the device status word (must match RMSNORM_DEVSTATUS_* in rmsnorm.h).
constexpr unsigned int DEVSTATUS_WAIT_TIMEOUT = 1u;

// Default budget of one bounded wait, in SM clock cycles (about a second at
// the GB300's ~2 GHz SM clock).
constexpr long long DEFAULT_WAIT_BUDGET = 2000000000LL;

// ---------------------------------------------------------------------------
// fp16 / bf16 <-> fp32.  Eight 16-bit values travel as one uint4.
// ---------------------------------------------------------------------------
template <typename T> struct Cvt;

template <> struct Cvt<__half> {
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        __half2 h;
        memcpy(&h, &u, 4);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);  // each rounded to nearest even
        uint32_t u;
        memcpy(&u, &h, 4);
        return u;
    }
    static __device__ __forceinline__ float load1(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void store1(__half *p, float v) { *p = __float2half_rn(v); }
};

template <> struct Cvt<__nv_bfloat16> {
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        __nv_bfloat162 h;
        memcpy(&h, &u, 4);
        return __bfloat1622float2(h);
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // each rounded to nearest even
        uint32_t u;
        memcpy(&u, &h, 4);
        return u;
    }
    static __device__ __forceinline__ float load1(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store1(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

template <> struct Cvt<float> {
    static __device__ __forceinline__ float load1(const float *p) { return *p; }
    static __device__ __forceinline__ void store1(float *p, float v) { *p = v; }
};

// Elements of T in one 16-byte vector, and the float2 pairs they fill.
template <typename T> __host__ __device__ constexpr int vec_elems() { return 16 / (int)sizeof(T); }
template <typename T> __host__ __device__ constexpr int vec_pairs() { return 8 / (int)sizeof(T); }

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
    float2 a = Cvt<T>::unpack2(v.x), b = Cvt<T>::unpack2(v.y);
    float2 c = Cvt<T>::unpack2(v.z), d = Cvt<T>::unpack2(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float f[8]) {
    uint4 v;
    v.x = Cvt<T>::pack2(f[0], f[1]);
    v.y = Cvt<T>::pack2(f[2], f[3]);
    v.z = Cvt<T>::pack2(f[4], f[5]);
    v.w = Cvt<T>::pack2(f[6], f[7]);
    return v;
}

// Eight 16-bit values <-> four float2 (the operand shape of the packed fp32x2
// arithmetic below).
template <typename T>
__device__ __forceinline__ void unpack8(const uint4 &v, float2 f[4]) {
    f[0] = Cvt<T>::unpack2(v.x);
    f[1] = Cvt<T>::unpack2(v.y);
    f[2] = Cvt<T>::unpack2(v.z);
    f[3] = Cvt<T>::unpack2(v.w);
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float2 f[4]) {
    uint4 v;
    v.x = Cvt<T>::pack2(f[0].x, f[0].y);
    v.y = Cvt<T>::pack2(f[1].x, f[1].y);
    v.z = Cvt<T>::pack2(f[2].x, f[2].y);
    v.w = Cvt<T>::pack2(f[3].x, f[3].y);
    return v;
}

// One 16-byte vector of T <-> fp32, as float2 pairs (fp16/bf16: four pairs,
// fp32: two) or as plain floats (eight or four).
template <typename T>
__device__ __forceinline__ void unpack_vec(const uint4 &v, float2 (&f)[vec_pairs<T>()]) {
    if constexpr (sizeof(T) == 4) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    } else {
        unpack8<T>(v, f);
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack_vec(const float2 (&f)[vec_pairs<T>()]) {
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                          __float_as_uint(f[1].y));
    } else {
        return pack8<T>(f);
    }
}

template <typename T>
__device__ __forceinline__ void unpack_vec(const uint4 &v, float (&f)[vec_elems<T>()]) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    } else {
        unpack8<T>(v, f);
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack_vec(const float (&f)[vec_elems<T>()]) {
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    } else {
        return pack8<T>(f);
    }
}

// Packed fp32x2 arithmetic (one instruction for two lanes of work on sm_100+),
// each result rounded to nearest even exactly as the scalar operation would be.
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Streaming 16-byte global load (evict-first: every byte is read once) and a
// plain 16-byte store.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_global(uint4 *p, const uint4 &v) { *p = v; }

// ---------------------------------------------------------------------------
// Sums in a fixed order.  The xor butterfly leaves the same bits in every
// lane (each step adds the same two operands in both lanes of a pair).
// ---------------------------------------------------------------------------
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D TMA bulk copy (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of the phase with the given parity (try_wait may suspend
// the thread for a while; test_wait returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// One arrival on an mbarrier of this CTA (release: this thread's earlier
// shared-memory accesses are ordered before it).
__device__ __forceinline__ void mbar_arrive_local(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits for the phase of `bar` with the given parity to complete; gives up
// after `budget` SM clock cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > budget) return false;
    }
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream finishes;
// it must wait here before touching anything that kernel wrote (a no-op when
// launched normally).  The previous kernel signals early with
// griddep_launch_dependents(); the wait still covers all of its writes.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Global -> shared 2-D tensor copy of one box of the tensor map at `tmap` (a
// kernel parameter's address) with its first element at column x (in the
// map's units; x times the unit size a multiple of 16 bytes), row y; rows past the tensor's end are
// zero-filled and still count toward the box's bytes on `bar`.  dst must be
// 128-byte aligned.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

}  // namespace rmsn

namespace rmsn {

// ---------------------------------------------------------------------------
// Thread-block clusters (inline PTX): rank, the hardware cluster barrier, and
// distributed shared memory (another CTA's shared memory in the cluster).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives and waits (release /
// acquire: shared-memory writes before it are visible to the cluster after).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of this CTA's shared variable at `p` in the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void dsmem_store_f2(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
                 : "memory");
}

// Asynchronous store of a float2 into another CTA's shared memory (addr, a
// shared::cluster address) that completes 8 bytes of the transaction count
// of that CTA's mbarrier (bar, a shared::cluster address) when it lands.
// Unlike an arrival with release semantics, it does not wait for this
// thread's earlier global writes to become visible first.
__device__ __forceinline__ void dsmem_store_async_f2(uint32_t addr, float2 v, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            addr),
        "f"(v.x), "f"(v.y), "r"(bar)
        : "memory");
}

// 16-byte load from a shared::cluster address (this or another CTA of the
// cluster).
__device__ __forceinline__ float4 dsmem_load_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// One arrival on an mbarrier in another CTA of the cluster, ordered after
// this thread's earlier (shared::cluster) writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
                 : "memory");
}

// try_wait that acquires at cluster scope (sees the writes that other CTAs
// ordered before their arrivals).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity,
                                                          long long budget) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock64() - t0 > budget) return false;
    }
}

}  // namespace rmsn
