// rope.cu -- rotary embedding of q and k fused with the KV-cache append
// ("Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
// Background, second bullet, and Task item 3: one kernel rotates q and k and
// writes k and v into the cache slab or a paged pool block, with cos/sin
// from a precomputed table or computed on the fly).
//
// Vectorised shapes (Dh % 16 == 0, 16-byte aligned, up to 32 rotation units
// per head) run warp-wide: a warp takes one token (or one of up to eight parts
// of it, when there are fewer tokens than warps), each lane owns one rotation
// unit -- 8 pairs, two 16-byte vectors, in the rotate-half layout; 4 pairs,
// one vector, interleaved -- of 32 / units heads at a time, and computes (or
// reads) the cos/sin of its own pairs once for all of that token's q and k
// heads.  No shared-memory table and no CTA barrier: every warp streams on
// its own, several heads' loads in flight per lane.  Other shapes take a
// CTA-wide kernel: persistent CTAs walk groups of four consecutive tokens,
// fill a shared-memory table of the Dh/2 (cos, sin) pairs of each token's
// position, and then rotate every q and k head of those tokens with it
// (element-wise, or with vectors for Dh past the warp kernel's limit); v is
// copied.
//
// On-the-fly angles without FP64 on the device: theta_i = p * base^(-2i/Dh).
// base^(-2i/Dh) is computed on the host in double (cached per thread for the
// last base and Dh) and split into a hi + lo pair of floats passed with the
// launch; per token p * (hi + lo) is formed as a double-float
// (an exact product error from fmaf), reduced modulo 2 pi with 2 pi split in
// two floats (Cody-Waite reduction): about 1e-8 rad of error at p = 1e6,
// where a plain float product is off by up to 0.06 rad.  The reduced angle
// lies in [-pi, pi], where the SFU's sine and cosine (__sincosf) are within
// about 2^-21 absolute; they replace sincosf, whose instruction count sat on
// every token's critical path (65536 tokens: 5869 -> 6142 GB/s).
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
// The warp kernel: two CTAs per SM leave 128 registers for four heads' loads
// in flight per lane.  Measured against three CTAs with two heads: +21 % at
// 4096 tokens, +6 % at 8192, +3 % at 16384, -1 % at 65536.
constexpr int ROPE_WARP_CTAS_PER_SM = 2;
constexpr int ROPE_HEADS_PER_BATCH = 4;   // heads whose loads a lane keeps in flight
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

// One rotation unit: PPU pairs of the head at src rotated into dst with the
// lane's (cos, sin) pairs cs, from registers xa (and xb, rotate-half: the
// vector half a head further on).
template <typename T, bool INTERLEAVED>
__device__ __forceinline__ void rotate_store(const uint4 &xa, const uint4 &xb, const float2 *cs,
                                             T *dst, int half) {
    if constexpr (!INTERLEAVED) {
        float2 a1[4], a2[4], y1[4], y2[4];
        unpack8<T>(xa, a1);
        unpack8<T>(xb, a2);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 c0 = cs[2 * m], c1 = cs[2 * m + 1];
            y1[m] = make_float2(a1[m].x * c0.x - a2[m].x * c0.y, a1[m].y * c1.x - a2[m].y * c1.y);
            y2[m] = make_float2(a2[m].x * c0.x + a1[m].x * c0.y, a2[m].y * c1.x + a1[m].y * c1.y);
        }
        *reinterpret_cast<uint4 *>(dst) = pack8<T>(y1);
        *reinterpret_cast<uint4 *>(dst + half) = pack8<T>(y2);
    } else {
        float2 x[4], y[4];
        unpack8<T>(xa, x);
#pragma unroll
        for (int m = 0; m < 4; ++m)
            y[m] = make_float2(x[m].x * cs[m].x - x[m].y * cs[m].y, x[m].y * cs[m].x + x[m].x * cs[m].y);
        *reinterpret_cast<uint4 *>(dst) = pack8<T>(y);
    }
}

// Rotates heads [0, H) of one token (src -> dst, head stride Dh): this lane's
// unit of heads h_first, h_first + step, ...; ROPE_HEADS_PER_BATCH heads'
// loads are issued before any of them is stored (heads never share an
// address, so in place too).
template <typename T, bool INTERLEAVED>
__device__ __forceinline__ void rotate_heads(const T *src, T *dst, int H, int h_first, int step,
                                             int Dh, int unit_off, const float2 *cs) {
    constexpr int HB = ROPE_HEADS_PER_BATCH;
    const int half = Dh / 2;
    for (int h0 = h_first; h0 < H; h0 += HB * step) {
        uint4 xa[HB], xb[HB];
#pragma unroll
        for (int b = 0; b < HB; ++b) {
            const int h = h0 + b * step;
            if (h < H) {
                const T *sp = src + (int64_t)h * Dh + unit_off;
                xa[b] = *reinterpret_cast<const uint4 *>(sp);
                if constexpr (!INTERLEAVED) xb[b] = *reinterpret_cast<const uint4 *>(sp + half);
                else xb[b] = xa[b];
            }
        }
#pragma unroll
        for (int b = 0; b < HB; ++b) {
            const int h = h0 + b * step;
            if (h < H) rotate_store<T, INTERLEAVED>(xa[b], xb[b], cs, dst + (int64_t)h * Dh + unit_off, half);
        }
    }
}

template <typename T, bool INTERLEAVED>
__global__ void __launch_bounds__(ROPE_NT, ROPE_WARP_CTAS_PER_SM) rope_warp_kernel(const RopeArgs a,
                                                                                 int wpt) {
    constexpr int PPU = INTERLEAVED ? 4 : 8;  // rotation pairs per unit
    __shared__ float2 s_inv[ROPE_MAX_DH / 2];
    const int Dh = a.Dh, half = Dh / 2;
    const bool table = a.cos_sin != nullptr;
    if (!table) {  // the lanes of a warp read different frequencies: from shared memory
        for (int i = threadIdx.x; i < half; i += ROPE_NT) s_inv[i] = a.inv[i];
        __syncthreads();
    }
    griddep_wait();  // programmatic dependent: no global access before this

    const int lane = threadIdx.x & 31;
    const int units = half / PPU;      // per head, at most 32 here
    const int hpi = 32 / units;        // heads a warp covers per step
    const int hs = lane / units, c = lane - hs * units;
    const bool rot_lane = hs < hpi;
    const int unit_off = INTERLEAVED ? c * 8 : c * PPU;  // first element of the unit
    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const uint4 *v = static_cast<const uint4 *>(a.v);
    T *q_out = static_cast<T *>(a.q_out);
    T *k_cache = static_cast<T *>(a.k_cache);
    uint4 *v_cache = static_cast<uint4 *>(a.v_cache);
    const int Hq = a.Hq, Hkv = a.Hkv;
    const int v_vecs = Hkv * Dh / 8;   // 16-byte vectors of v per token

    const int64_t n_items = a.T * wpt;
    const int64_t n_warps = (int64_t)gridDim.x * (ROPE_NT / 32);
    for (int64_t w = ((int64_t)blockIdx.x * ROPE_NT + threadIdx.x) >> 5; w < n_items; w += n_warps) {
        const int64_t t = w / wpt;
        const int part = (int)(w - t * wpt);
        const int64_t p = a.positions[t];
        const int64_t slot = a.slots[t];
        const bool pos_ok = p >= 0 && (!table || p < a.max_pos);
        const bool slot_ok = slot < a.num_slots;  // negative: not written
        if ((!pos_ok || !slot_ok) && lane == 0 && part == 0) atomicOr(a.status, DEVSTATUS_BAD_INDEX);
        if (!pos_ok) continue;
        const bool write_kv = slot_ok && slot >= 0;

        float2 cs[PPU];
        if (rot_lane) {
            const int i0 = c * PPU;
            if (table) {
                const float4 *row = reinterpret_cast<const float4 *>(a.cos_sin + p * Dh);
#pragma unroll
                for (int m = 0; m < PPU; m += 4) {
                    const float4 cv = row[(i0 + m) / 4], sv = row[(half + i0 + m) / 4];
                    cs[m] = make_float2(cv.x, sv.x);
                    cs[m + 1] = make_float2(cv.y, sv.y);
                    cs[m + 2] = make_float2(cv.z, sv.z);
                    cs[m + 3] = make_float2(cv.w, sv.w);
                }
            } else {
#pragma unroll
                for (int m = 0; m < PPU; ++m) {
                    const float2 f = s_inv[i0 + m];
                    __sincosf(reduced_angle(p, f.x, f.y), &cs[m].y, &cs[m].x);
                }
            }
            const int step = wpt * hpi;
            rotate_heads<T, INTERLEAVED>(q + t * Hq * (int64_t)Dh, q_out + t * Hq * (int64_t)Dh, Hq,
                                         part * hpi + hs, step, Dh, unit_off, cs);
            if (write_kv)
                rotate_heads<T, INTERLEAVED>(k + t * Hkv * (int64_t)Dh,
                                             k_cache + slot * Hkv * (int64_t)Dh, Hkv,
                                             part * hpi + hs, step, Dh, unit_off, cs);
        }
        if (write_kv) {
            const uint4 *vs = v + t * v_vecs;
            uint4 *vd = v_cache + slot * v_vecs;
            for (int i = part * 32 + lane; i < v_vecs; i += 2 * 32 * wpt) {
                const int i2 = i + 32 * wpt;
                const uint4 x1 = vs[i];
                uint4 x2 = x1;
                if (i2 < v_vecs) x2 = vs[i2];
                vd[i] = x1;
                if (i2 < v_vecs) vd[i2] = x2;
            }
        }
    }
    griddep_launch_dependents();
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
                    __sincosf(reduced_angle(p, a.inv[i].x, a.inv[i].y), &sn, &c);
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
cudaError_t launch_rope_t(const RopeArgs &a, bool vec, int sm, cudaStream_t s) {
    const int64_t resident = (int64_t)sm * ROPE_CTAS_PER_SM;
    const int units = INTERLEAVED ? a.Dh / 8 : a.Dh / 16;  // rotation units per head
    // At every token count: replayed from a CUDA graph, 8 tokens take 3.3 us
    // here against 5.1 us with the CTA-wide kernel (1 token: 3.2 us either).
    if (vec && units <= 32) {
        // warps per token: spread a few tokens over more warps (up to 8)
        const int64_t resident_w = (int64_t)sm * ROPE_WARP_CTAS_PER_SM;
        const int64_t warps = resident_w * (ROPE_NT / 32);
        const int wpt = (int)std::max<int64_t>(1, std::min<int64_t>(8, warps / a.T));
        const int64_t need = (a.T * wpt + ROPE_NT / 32 - 1) / (ROPE_NT / 32);
        const int grid = (int)std::min<int64_t>(need, resident_w);
        return launch_pdl(rope_warp_kernel<T, INTERLEAVED>, dim3(grid), dim3(ROPE_NT), 0, s, a, wpt);
    }
    const int64_t groups = (a.T + ROPE_TOKENS_PER_ITER - 1) / ROPE_TOKENS_PER_ITER;
    const int grid = (int)std::min<int64_t>(groups, resident);
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
    const bool vec = Dh % 16 == 0 && al16(q) && al16(q_out) && (!cos_sin || al16(cos_sin)) &&
                     (Hkv == 0 || (al16(k) && al16(v) && al16(k_cache) && al16(v_cache)));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == RMSNORM_F16)
        e = interleaved ? launch_rope_t<__half, true>(a, vec, sm, s)
                        : launch_rope_t<__half, false>(a, vec, sm, s);
    else
        e = interleaved ? launch_rope_t<__nv_bfloat16, true>(a, vec, sm, s)
                        : launch_rope_t<__nv_bfloat16, false>(a, vec, sm, s);
    return e == cudaSuccess ? RMSNORM_OK : record_cuda_error(e);
}
