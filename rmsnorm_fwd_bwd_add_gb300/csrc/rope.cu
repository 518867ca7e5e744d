// rope.cu -- rotary embedding of q and k fused with the KV-cache append
// ("Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
// Background, second bullet, and Task item 3: one kernel rotates q and k and
// writes k and v into the cache slab or a paged pool block, with cos/sin
// from a precomputed table or computed on the fly).
//
// Persistent CTAs walk groups of four consecutive tokens.  For each group the
// CTA first fills a shared-memory table of the Dh/2 (cos, sin) pairs of each
// token's position -- read from the caller's table or computed -- and then
// every q and k head of those tokens rotates with it; v is copied.  Vectorised threads own 8 rotation pairs each
// (two 16-byte vectors in the rotate-half layout, one in the interleaved one).
//
// On-the-fly angles without FP64 on the device: theta_i = p * base^(-2i/Dh).
// base^(-2i/Dh) is computed on the host in double (cached per thread for the
// last base and Dh) and split into a hi + lo pair of floats passed with the
// launch; per token p * (hi + lo) is formed as a double-float
// (an exact product error from fmaf), reduced modulo 2 pi with 2 pi split in
// two floats (Cody-Waite reduction), and sincosf takes the reduced angle:
// about 1e-8 rad of error at p = 1e6, where a plain float product is off by
// up to 0.06 rad.
//
// Device data is validated: a position outside the table (or negative) or a
// slot past the cache sets RMSNORM_DEVSTATUS_BAD_INDEX and that token's
// affected outputs are skipped; nothing is read or written out of range.
#include "rmsnorm.h"

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "launch_util.h"

namespace rmsn {
int current_sm_count(int *sm);
int current_status_word(unsigned int **status);
int record_cuda_error(cudaError_t e);
}  // namespace rmsn

namespace {

using namespace rmsn;

constexpr int ROPE_NT = 256;
constexpr int ROPE_CTAS_PER_SM = 4;
constexpr int ROPE_MAX_DH = 1024;
constexpr int ROPE_TOKENS_PER_ITER = 4;  // tokens a CTA handles between barriers
constexpr unsigned int DEVSTATUS_BAD_INDEX = 2u;

constexpr double TWO_PI = 6.283185307179586476925286766559;
constexpr float TWO_PI_HI = (float)TWO_PI;
constexpr float TWO_PI_LO = (float)(TWO_PI - (double)TWO_PI_HI);
constexpr float INV_TWO_PI = (float)(1.0 / TWO_PI);

struct RopeArgs {
    float2 inv[ROPE_MAX_DH / 2];  // (hi, lo) floats of base^(-2i/Dh), from the host in double
    const void *q, *k, *v;
    const int64_t *positions, *slots;
    void *q_out, *k_cache, *v_cache;
    const float *cos_sin;  // [max_pos, Dh]: Dh/2 cosines then Dh/2 sines, or null
    int64_t max_pos;
    float base;
    int64_t T, num_slots;
    int Hq, Hkv, Dh;
    unsigned int *status;
};

// p * inv as a double-float, reduced to about [-pi, pi].
__device__ __forceinline__ float reduced_angle(int64_t p, float inv_hi, float inv_lo) {
    const float ph = (float)p;
    const float pl = (float)(p - (int64_t)ph);  // exact: the part of p a float cannot hold
    const float s = ph * inv_hi;
    const float e = fmaf(ph, inv_hi, -s);  // exact error of that product
    const float t = fmaf(ph, inv_lo, fmaf(pl, inv_hi, e));
    const float kq = rintf(s * INV_TWO_PI);
    float r = fmaf(-kq, TWO_PI_HI, s);
    r = fmaf(-kq, TWO_PI_LO, r);
    return r + t;
}

template <typename T, bool INTERLEAVED, bool VEC>
__global__ void __launch_bounds__(ROPE_NT, ROPE_CTAS_PER_SM) rope_kv_kernel(const RopeArgs a) {
    constexpr int TPI = ROPE_TOKENS_PER_ITER;
    __shared__ float2 cs[TPI][ROPE_MAX_DH / 2];   // (cos, sin) of the group's tokens
    __shared__ int64_t s_slot[TPI];
    __shared__ int s_flags[TPI];                  // bit 0: position valid, bit 1: write k/v
    const int tid = threadIdx.x;
    const int Dh = a.Dh, half = Dh / 2;
    const bool table = a.cos_sin != nullptr;
    griddep_wait();  // programmatic dependent: no global access before this

    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    T *q_out = static_cast<T *>(a.q_out);
    T *k_cache = static_cast<T *>(a.k_cache);
    T *v_cache = static_cast<T *>(a.v_cache);
    // work items per token: rotation units of q heads, then of k heads, then
    // v units (VEC: a unit is 8 pairs / one 16-byte vector; else one pair /
    // one element)
    constexpr int PAIRS = VEC ? (INTERLEAVED ? 4 : 8) : 1;
    const int rot_units = half / PAIRS;
    const int v_units = VEC ? Dh / 8 : Dh;
    const int nq = a.Hq * rot_units, nk = a.Hkv * rot_units, nv = a.Hkv * v_units;
    const int per_token = nq + nk + nv;

    // CTA b takes the groups of TPI consecutive tokens b, b + grid, ...
    for (int64_t t0 = (int64_t)blockIdx.x * TPI; t0 < a.T; t0 += (int64_t)gridDim.x * TPI) {
        if (tid < TPI) {
            const int64_t t = t0 + tid;
            int flags = 0;
            int64_t slot = -1;
            if (t < a.T) {
                const int64_t p = a.positions[t];
                slot = a.slots[t];
                const bool pos_ok = p >= 0 && (!table || p < a.max_pos);
                const bool slot_ok = slot < a.num_slots;  // negative: not written
                if (!pos_ok || !slot_ok) atomicOr(a.status, DEVSTATUS_BAD_INDEX);
                flags = (pos_ok ? 1 : 0) | (pos_ok && slot_ok && slot >= 0 ? 2 : 0);
            }
            s_slot[tid] = slot;
            s_flags[tid] = flags;
        }
        __syncthreads();
        for (int e = tid; e < TPI * half; e += ROPE_NT) {
            const int j = e / half, i = e - j * half;
            if (s_flags[j] & 1) {
                const int64_t p = a.positions[t0 + j];
                float c, sn;
                if (table) {
                    c = a.cos_sin[p * Dh + i];
                    sn = a.cos_sin[p * Dh + half + i];
                } else {
                    sincosf(reduced_angle(p, a.inv[i].x, a.inv[i].y), &sn, &c);
                }
                cs[j][i] = make_float2(c, sn);
            }
        }
        __syncthreads();
        for (int e = tid; e < TPI * per_token; e += ROPE_NT) {
            const int j = e / per_token, it = e - j * per_token;
            const int flags = s_flags[j];
            if (!(flags & 1) || (it >= nq && !(flags & 2))) continue;
            const int64_t t = t0 + j;
            const int64_t slot = s_slot[j];
            const float2 *csj = cs[j];
            if (it < nq + nk) {
                const bool is_q = it < nq;
                const int u = is_q ? it : it - nq;
                const int h = u / rot_units, c = u % rot_units;
                const T *src = is_q ? q + (t * a.Hq + h) * (int64_t)Dh : k + (t * a.Hkv + h) * (int64_t)Dh;
                T *dst = is_q ? q_out + (t * a.Hq + h) * (int64_t)Dh
                              : k_cache + (slot * a.Hkv + h) * (int64_t)Dh;
                if constexpr (VEC && !INTERLEAVED) {
                    const int i0 = c * 8;
                    float2 x1[4], x2[4], y1[4], y2[4];
                    unpack8<T>(*reinterpret_cast<const uint4 *>(src + i0), x1);
                    unpack8<T>(*reinterpret_cast<const uint4 *>(src + half + i0), x2);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 c0 = csj[i0 + 2 * m], c1 = csj[i0 + 2 * m + 1];
                        y1[m] = make_float2(x1[m].x * c0.x - x2[m].x * c0.y, x1[m].y * c1.x - x2[m].y * c1.y);
                        y2[m] = make_float2(x2[m].x * c0.x + x1[m].x * c0.y, x2[m].y * c1.x + x1[m].y * c1.y);
                    }
                    *reinterpret_cast<uint4 *>(dst + i0) = pack8<T>(y1);
                    *reinterpret_cast<uint4 *>(dst + half + i0) = pack8<T>(y2);
                } else if constexpr (VEC && INTERLEAVED) {
                    const int j0 = c * 8;  // elements j0..j0+7 = pairs c*4 .. c*4+3
                    float2 x[4], y[4];
                    unpack8<T>(*reinterpret_cast<const uint4 *>(src + j0), x);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 cc = csj[c * 4 + m];
                        y[m] = make_float2(x[m].x * cc.x - x[m].y * cc.y, x[m].y * cc.x + x[m].x * cc.y);
                    }
                    *reinterpret_cast<uint4 *>(dst + j0) = pack8<T>(y);
                } else {
                    const int ia = INTERLEAVED ? 2 * c : c;
                    const int ib = INTERLEAVED ? 2 * c + 1 : c + half;
                    const float xa = Cvt<T>::load1(src + ia), xb = Cvt<T>::load1(src + ib);
                    const float2 cc = csj[c];
                    Cvt<T>::store1(dst + ia, xa * cc.x - xb * cc.y);
                    Cvt<T>::store1(dst + ib, xb * cc.x + xa * cc.y);
                }
            } else {
                const int u = it - nq - nk;
                const int h = u / v_units, c = u % v_units;
                const T *src = v + (t * a.Hkv + h) * (int64_t)Dh;
                T *dst = v_cache + (slot * a.Hkv + h) * (int64_t)Dh;
                if constexpr (VEC)
                    reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
                else
                    dst[c] = src[c];
            }
        }
        __syncthreads();  // cs, s_slot and s_flags are rewritten for the next group
    }
    griddep_launch_dependents();
}

template <typename T, bool INTERLEAVED>
cudaError_t launch_rope_t(const RopeArgs &a, bool vec, int grid, cudaStream_t s) {
    if (vec)
        return launch_pdl(rope_kv_kernel<T, INTERLEAVED, true>, dim3(grid), dim3(ROPE_NT), 0, s, a);
    return launch_pdl(rope_kv_kernel<T, INTERLEAVED, false>, dim3(grid), dim3(ROPE_NT), 0, s, a);
}

// base^(-2i/Dh) for i < Dh/2 as (hi, lo) float pairs; the last (base, Dh) of
// the calling thread is kept, as a model calls with the same pair every layer.
void inverse_frequencies(float base, int Dh, float2 *inv) {
    thread_local float last_base = -1.f;
    thread_local int last_dh = -1;
    thread_local float2 last[ROPE_MAX_DH / 2];
    if (base != last_base || Dh != last_dh) {
        for (int i = 0; i < Dh / 2; ++i) {
            const double f = std::pow((double)base, -2.0 * (double)i / (double)Dh);
            const float hi = (float)f;
            last[i] = make_float2(hi, (float)(f - (double)hi));
        }
        last_base = base;
        last_dh = Dh;
    }
    std::copy(last, last + Dh / 2, inv);
}

bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" int rmsnorm_rope_kv_append(const void *q, const void *k, const void *v,
                                      const int64_t *positions, const int64_t *slots, void *q_out,
                                      void *k_cache, void *v_cache, const float *cos_sin,
                                      int64_t max_pos, float rope_base, int interleaved, int64_t T,
                                      int64_t Hq, int64_t Hkv, int64_t Dh, int64_t num_slots,
                                      int dtype, void *stream) {
    if (dtype != RMSNORM_F16 && dtype != RMSNORM_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (T < 0 || Hq < 0 || Hkv < 0 || num_slots < 0 || Dh <= 0 || Dh % 2) return RMSNORM_ERR_INVALID_ARG;
    if (Dh > ROPE_MAX_DH || Hq > (1 << 16) || Hkv > (1 << 16)) return RMSNORM_ERR_UNSUPPORTED;
    if (cos_sin ? max_pos <= 0 : !(rope_base > 0.f && rope_base < 3.0e38f)) return RMSNORM_ERR_INVALID_ARG;
    if (T == 0) return RMSNORM_OK;
    if (!positions || !slots || (Hq > 0 && (!q || !q_out)) ||
        (Hkv > 0 && (!k || !v || !k_cache || !v_cache)))
        return RMSNORM_ERR_INVALID_ARG;
    if (T > INT64_MAX / ((Hq + 2 * Hkv + 1) * Dh * 2) || num_slots > INT64_MAX / (Hkv * Dh * 2 + 1))
        return RMSNORM_ERR_UNSUPPORTED;
    const size_t nq = (size_t)T * Hq * Dh * 2, nkv = (size_t)T * Hkv * Dh * 2;
    const size_t nc = (size_t)num_slots * Hkv * Dh * 2;
    // q_out may be q itself; the caches must not overlap the inputs, q_out or
    // each other
    if (q_out != q && overlap(q_out, nq, q, nq)) return RMSNORM_ERR_INVALID_ARG;
    const void *ins[] = {q, k, v};
    const size_t nins[] = {nq, nkv, nkv};
    for (int i = 0; i < 3; ++i) {
        if (overlap(k_cache, nc, ins[i], nins[i]) || overlap(v_cache, nc, ins[i], nins[i]))
            return RMSNORM_ERR_INVALID_ARG;
        if (i > 0 && overlap(q_out, nq, ins[i], nins[i])) return RMSNORM_ERR_INVALID_ARG;
    }
    if (overlap(k_cache, nc, v_cache, nc) || overlap(k_cache, nc, q_out, nq) ||
        overlap(v_cache, nc, q_out, nq))
        return RMSNORM_ERR_INVALID_ARG;

    int sm = 0;
    unsigned int *status = nullptr;
    int st = current_sm_count(&sm);
    if (st == RMSNORM_OK) st = current_status_word(&status);
    if (st != RMSNORM_OK) return st;
    static_assert(sizeof(RopeArgs) < 8192, "kernel parameters stay small");
    RopeArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.positions = positions; a.slots = slots;
    a.q_out = q_out; a.k_cache = k_cache; a.v_cache = v_cache;
    a.cos_sin = cos_sin; a.max_pos = max_pos; a.base = rope_base;
    a.T = T; a.num_slots = num_slots;
    a.Hq = (int)Hq; a.Hkv = (int)Hkv; a.Dh = (int)Dh;
    a.status = status;
    if (!cos_sin) inverse_frequencies(rope_base, (int)Dh, a.inv);
    const bool vec = Dh % 16 == 0 && al16(q) && al16(q_out) && (Hkv == 0 ||
                     (al16(k) && al16(v) && al16(k_cache) && al16(v_cache)));
    const int64_t groups = (T + ROPE_TOKENS_PER_ITER - 1) / ROPE_TOKENS_PER_ITER;
    const int grid = (int)std::min<int64_t>(groups, (int64_t)sm * ROPE_CTAS_PER_SM);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == RMSNORM_F16)
        e = interleaved ? launch_rope_t<__half, true>(a, vec, grid, s)
                        : launch_rope_t<__half, false>(a, vec, grid, s);
    else
        e = interleaved ? launch_rope_t<__nv_bfloat16, true>(a, vec, grid, s)
                        : launch_rope_t<__nv_bfloat16, false>(a, vec, grid, s);
    return e == cudaSuccess ? RMSNORM_OK : record_cuda_error(e);
}
