// staged.cuh -- persistent RMSNorm kernels that stage rows through a shared
// memory ring with the 1-D TMA bulk copy (cp.async.bulk + mbarrier).
//
// Work unit: a tile of `tile_rows` consecutive rows.  Dense rows make one
// tile of one tensor ONE bulk copy.  CTA b owns tiles b, b + grid, b + 2*grid,
// ... (a static assignment, so the VJP's gw partials are summed in the same
// order on every run).  Thread 0 keeps `stages` tiles in flight; every thread
// waits on the tile's mbarrier, converts its vectors of the row from shared
// memory into fp32 registers once, and writes its outputs straight to global
// memory.  A 16-byte vector holds eight fp16/bf16 or four fp32 elements.
//
// GEN = true is the general instance: rows a stride apart (in the sub-warp
// shape a tensor whose tile is not contiguous is copied one row at a time,
// those copies spread over all threads of the CTA; the tile is dense in
// shared memory either way)
// and the per-row scale rstd (written by the forward, read by the VJP in place
// of its own sum of squares).  GEN = false is the dense instance without
// rstd; the launcher picks it whenever it applies, so the common case carries
// none of the general case's address arithmetic or registers.
//
// Two shapes of work inside a tile:
//   * G == NT ("CTA per row", D > 1024): one row per tile; each thread owns
//     V vectors of 8 elements; sum of squares = warp shuffle tree, then the
//     warp totals (read one per lane from shared memory) summed by a second
//     shuffle tree: the warp-then-block reduction of the fused-norm design,
//     one CTA barrier per row.  A stage is handed back to the producer one row
//     later, at the next barrier, when every thread is done with it.
//   * G <= 32 ("sub-warp / warp per row", D <= 1024): NT/G rows at a time,
//     each reduced by a G-lane shuffle tree only; no shared-memory reduction,
//     so no multi-warp band exists to get wrong.
// A thread multiplies by the same weight columns in every row it touches
// (fixed column ownership): w' = weight_bias + w is converted to fp32 once per
// CTA, and the VJP's gw contributions stay in the owning thread's registers.
// Per-element arithmetic is packed fp32x2.
//
// Sources: "Fused residual-add RMSNorm and fused RoPE + KV-append decode
// kernels", Background (FusedAddRMSNorm: one pass, fp32 sum kept once,
// warp-then-block sum of squares, weight_bias, two outputs); "RMSNormVJP
// backward writes a full {n_rows, D} gw_temp intermediate", Proposed changes
// (reduce gw across rows inside the kernel, no {n_rows, D} temporary).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

template <typename T, int MODE, int NT, int G, int V, int MINB, bool GEN, bool SH, bool CLAIM>
__global__ void __launch_bounds__(NT, MINB) staged_kernel(const __grid_constant__ KernelArgs a) {
    constexpr int NWARPS = NT / 32;
    constexpr int WP = NWARPS <= 4 ? 4 : NWARPS <= 8 ? 8 : NWARPS <= 16 ? 16 : 32;
    constexpr int NG = NT / G;  // rows processed side by side
    constexpr int VP = vec_pairs<T>();   // float2 pairs per 16-byte vector
    constexpr int EPV = vec_elems<T>();  // elements per 16-byte vector
    constexpr bool CTA_ROW = (G == NT);
    // Tiles of several rows a stride apart take one copy per row, spread over
    // the CTA's threads; a CTA-per-row tile is always a single copy.
    constexpr bool SPREAD_COPIES = GEN && !CTA_ROW;
    // Some VJP instances re-read a row from the stage for their outputs
    // instead of holding it in registers across the reduction (a CTA-per-row
    // stage is released only at the next row's barrier): those staged_reload
    // names, and the CTA-per-row VJPs of shifted rows whose register cap is
    // below 128 a thread, where the edge handling's registers would spill (D =
    // 4097 bf16, 320 threads: 8 bytes spilled when held, 86 registers re-read;
    // 4024 -> 4252 GB/s, 16384 rows).  With a cap of 128 they hold their rows
    // (110-112 registers; bf16, 16384 rows, rotating buffers: D = 4097 5358 ->
    // 5582 GB/s, D = 2052 4339 -> 4988, D = 8196 5779 -> 6165).
    constexpr bool RELOAD = staged_reload(MODE, NT, G, V) ||
                            (SH && is_vjp(MODE) && G == NT && NT * MINB > 512);
    constexpr int NTENS = input_tensors(MODE);
    constexpr bool VJP = is_vjp(MODE);
    constexpr bool ADD = (MODE == MODE_VJP_ADD);
    static_assert(G <= 32 || G == NT, "a row belongs to at most one warp, or to the whole CTA");
    static_assert(NWARPS <= 32, "one warp total per lane");
    static_assert(!(SH && GEN), "shifted rows are dense rows");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);   // [MAX_STAGES]
    int64_t *stage_tile = reinterpret_cast<int64_t *>(smem + 64);  // [MAX_STAGES] claimed tiles
    float2 *red = reinterpret_cast<float2 *>(smem + 128);  // [2][NWARPS]
    unsigned char *ring = smem + STAGED_HEADER_BYTES;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gid = tid / G;
    const int gl = tid % G;
    const int D = a.D;
    const int NV = D / EPV;
    const uint32_t row_bytes = (uint32_t)D * (uint32_t)sizeof(T);
    // SH ("shifted rows"): every row tensor's rows start at the same offset
    // from a 16-byte boundary, but not at 0 (an unaligned base, or D * size a
    // not multiple of 16).  Each row is copied as its 16-byte aligned
    // superset.  Its first `hd` elements (before the first boundary) and its
    // last ones (after the last whole vector) are the row's edge elements,
    // at most 14; between them lie NB whole, aligned vectors, which the
    // threads own exactly as they own an aligned row's vectors (the same
    // configuration; one vector on from the copy's start when the row is
    // offset).  Edge element i belongs to lane G - 1 - i of the row's group
    // (the CTA's last lanes), read and written one element at a time.  The
    // grid is a multiple of the offset's period in rows (and tiles of several
    // rows are multiples of 8 rows), so all of a thread's rows have the same
    // offset `shm`: its columns, its w' and its gw accumulators stay fixed.
    const uint32_t shm =
        SH ? (uint32_t)(((uintptr_t)a.in0 + (uint64_t)(CTA_ROW ? blockIdx.x : gid) * row_bytes) & 15u)
           : 0u;
    const int hd = SH && shm ? (int)((16u - shm) / sizeof(T)) : 0;  // head elements
    const int NB = SH ? (D - hd) / EPV : NV;                         // whole vectors
    const int bo = SH && shm ? 1 : 0;  // the copy's vector that holds whole vector 0
    constexpr int ES = !SH ? 1 : (G >= 16 ? 1 : 2);                 // edge elements a lane
    // Column of this lane's edge slot e, or -1.
    auto edge_col = [&](int e) -> int {
        const int i = (G - 1 - gl) + e * G;
        return (!SH || i >= D - NB * EPV) ? -1 : i < hd ? i : NB * EPV + i;
    };
    const int S = a.stages;
    const int TR = a.tile_rows;
    const int64_t rows = a.rows;
    const uint32_t SB = a.stage_bytes;
    const int64_t grid = gridDim.x;
    const int64_t nk = (a.num_tiles - (int64_t)blockIdx.x + grid - 1) / grid;  // >= 1
    // Claimed tiles: a forward may take most of its tiles from counters at
    // run time (a.tile_ctr) instead of the static round robin, so that every
    // CTA stays busy until the last tile is taken -- a CTA slowed down by the
    // memory system simply takes fewer.  The CTAs form K = a.claim_k groups
    // (CTA b in group b % K, K dividing the grid); group j owns tiles j, j +
    // K, j + 2K, ... and a counter of its own, so K counters share the
    // claims.  Each CTA's first S tiles are fixed (its ring fills with no
    // claim to wait for); after that it claims one tile at a time, one
    // refill ahead.  Rows of a forward are independent, so the results do
    // not depend on which CTA takes a row.  Not the VJP (a CTA's gw partial
    // row sums a fixed set of rows, which keeps gw's bits fixed), nor shifted
    // rows (a CTA's columns follow its rows' offset), nor tiles copied row by
    // row; and only in the CLAIM instances, so that the others run the static
    // loop with none of this compiled in (it cost the D = 8192 forward 2.5 %).
    constexpr bool DYN_OK = CLAIM && !VJP && !SH && !SPREAD_COPIES;
    const bool dyn = DYN_OK && a.tile_ctr != nullptr;
    const int CK = dyn ? a.claim_k : 1;                       // groups (counters)
    const int64_t c_home = (int64_t)blockIdx.x % CK;          // this CTA's group
    const int64_t c_rank = (int64_t)blockIdx.x / CK;          // its rank in the group
    const int64_t c_size = grid / CK;                         // CTAs of a group
    unsigned long long *c_ctr = dyn ? a.tile_ctr + CLAIM_STRIDE * c_home : nullptr;
    const float eps = a.eps;
    // 1/D once per CTA: the per-row means are products, not divisions (exact
    // for D a power of two; within an ulp of the quotient otherwise).
    const float inv_D = 1.0f / (float)D;

    const T *in0 = static_cast<const T *>(a.in0);
    const T *in1 = static_cast<const T *>(a.in1);
    const T *in2 = static_cast<const T *>(a.in2);
    uint4 *out0 = static_cast<uint4 *>(a.out0);
    uint4 *out1 = static_cast<uint4 *>(a.out1);
    // Output row strides in vectors.
    const int64_t lo0 = GEN ? a.ld_out0 / EPV : NV, lo1 = GEN ? a.ld_out1 / EPV : NV;

    auto stage_ptr = [&](int s, int tensor) -> unsigned char * {
        return ring + ((size_t)s * NTENS + tensor) * SB;
    };

    // ---- producer ----
    // Thread 0 posts a tile's expected bytes on its stage's mbarrier and
    // issues its copies.  With SPREAD_COPIES thread 0 posts the bytes before
    // the CTA barrier that ends the previous tile in that stage, and after the
    // barrier every thread issues a share of the tile's copies.
    int64_t issued = 0;  // tiles of this CTA issued so far (claimed: stages armed)
    int issue_stage = 0;
    bool exhausted = false;  // claimed tiles: the group's tiles have run out
    int64_t pending = 0;     // claimed tiles: the next claim, made a refill ahead
    auto more = [&]() -> bool { return dyn ? !exhausted : issued < nk; };
    // Thread 0, claimed tiles: the next tile of this CTA, or -1.  Group
    // index i (tile c_home + i * K): the CTA's first S are c_rank + s *
    // c_size, the rest S * c_size + the counter's next value.
    auto next_tile = [&]() -> int64_t {
        const bool fixed = issued < S;
        const int64_t gi = fixed ? c_rank + issued * c_size : (int64_t)S * c_size + pending;
        const int64_t t = c_home + gi * CK;
        if (t >= a.num_tiles) return -1;
        if (!fixed) pending = (int64_t)atomicAdd(c_ctr, 1ull);  // the next claim, ahead of need
        return t;
    };
    const uint64_t policy = l2_evict_first_policy();
    // First row and row count of this CTA's tile number idx; false for the
    // tile the test hook drops.
    auto tile_of = [&](int64_t idx, int64_t &row0, int &nr) -> bool {
        const int64_t t = (int64_t)blockIdx.x + idx * grid;
        row0 = t * TR;
        nr = (int)min((int64_t)TR, rows - row0);
        return t != a.drop_tile;
    };
    auto post_expect = [&](int64_t idx, int stage) {
        int64_t row0;
        int nr;
        if (tile_of(idx, row0, nr))
            mbar_arrive_expect_tx(&full[stage], (uint32_t)nr * row_bytes * NTENS);
    };
    // Copies first, first + step, ... of the tile's (tensor, row) pairs; a
    // tensor whose tile is contiguous goes as one copy, on its row 0's turn.
    auto issue_copies = [&](int64_t idx, int stage, int first, int step) {
        int64_t row0;
        int nr;
        if (!tile_of(idx, row0, nr)) return;
        for (int c = first; c < NTENS * nr; c += step) {
            const int tensor = c / nr, q = c - tensor * nr;
            const T *src = tensor == 0 ? in0 : tensor == 1 ? in1 : in2;
            const int64_t ld = tensor == 0 ? a.ld_in0 : tensor == 1 ? a.ld_in1 : a.ld_in2;
            unsigned char *dst = stage_ptr(stage, tensor);
            if (ld == D || nr == 1) {
                if (q == 0)
                    bulk_g2s(dst, src + row0 * ld, (uint32_t)nr * row_bytes, &full[stage], policy);
            } else {
                bulk_g2s(dst + (size_t)q * row_bytes, src + (row0 + q) * ld, row_bytes,
                         &full[stage], policy);
            }
        }
    };
    auto advance = [&]() {
        ++issued;
        issue_stage = issue_stage + 1 == S ? 0 : issue_stage + 1;
    };
    // General sub-warp tiles through the tensor maps (thread 0): one 2-D copy
    // per column box and tensor; a box past the last row is zero-filled and
    // its bytes still arrive, so the whole tile is expected.
    const int BC = SPREAD_COPIES ? a.box_cols : D;  // columns per box
    const bool tmap_mode = SPREAD_COPIES && a.use_tmap;
    auto issue_tmap = [&]() {
        const int64_t t = (int64_t)blockIdx.x + issued * grid;
        if (t != a.drop_tile) {
            uint64_t *bar = &full[issue_stage];
            const uint32_t box_bytes = (uint32_t)TR * (uint32_t)BC * (uint32_t)sizeof(T);
            const int nbox = D / BC;
            mbar_arrive_expect_tx(bar, box_bytes * (uint32_t)(nbox * NTENS));
            for (int tensor = 0; tensor < NTENS; ++tensor)
                for (int b = 0; b < nbox; ++b)
                    tma_load_2d(stage_ptr(issue_stage, tensor) + (size_t)b * box_bytes,
                                &a.tmap[tensor], b * BC * (int)sizeof(T) / 8, (int)(t * TR), bar,
                                policy);
        }
        advance();
    };
    // The tile starting at row0 (nr rows) of a dense tensor at `base`: its
    // first byte's offset from a 16-byte boundary (SH; 0 otherwise), and the
    // bytes of its copy (SH: the aligned superset).
    auto tile_off = [&](int64_t row0) -> uint32_t {
        return SH ? (uint32_t)(((uintptr_t)in0 + (uint64_t)row0 * row_bytes) & 15u) : 0u;
    };
    auto tile_bytes = [&](int nr, uint32_t off) -> uint32_t {
        return SH ? ((off + (uint32_t)nr * row_bytes + 15u) & ~15u) : (uint32_t)nr * row_bytes;
    };
    auto tile_src = [&](const T *base, int64_t row0, int64_t ld, uint32_t off) {
        return reinterpret_cast<const unsigned char *>(base + row0 * ld) - off;
    };
    auto issue_next = [&]() {  // thread 0, the whole tile
        int64_t row0;
        int nr;
        bool have;
        if (dyn) {
            const int64_t t = next_tile();
            if (t < 0) {  // none left: the stage's phase completes empty
                stage_tile[issue_stage] = -1;
                exhausted = true;
                mbar_arrive_local(&full[issue_stage]);
                advance();
                return;
            }
            stage_tile[issue_stage] = t;  // published by the arrival below
            row0 = t * TR;
            nr = (int)min((int64_t)TR, rows - row0);
            have = t != a.drop_tile;
        } else {
            have = tile_of(issued, row0, nr);
        }
        if (have) {
            uint64_t *bar = &full[issue_stage];
            if constexpr (!SPREAD_COPIES) {
                // dense tiles, or CTA per row (one row: one copy per tensor);
                // straight-line code, as thread 0 is on every row's critical path
                const uint32_t off = tile_off(row0);
                const uint32_t bytes = tile_bytes(nr, off);
                mbar_arrive_expect_tx(bar, bytes * NTENS);
                const int64_t l0 = GEN ? a.ld_in0 : D, l1 = GEN ? a.ld_in1 : D;
                const int64_t l2 = GEN ? a.ld_in2 : D;
                bulk_g2s(stage_ptr(issue_stage, 0), tile_src(in0, row0, l0, off), bytes, bar, policy);
                if constexpr (NTENS >= 2)
                    bulk_g2s(stage_ptr(issue_stage, 1), tile_src(in1, row0, l1, off), bytes, bar,
                             policy);
                if constexpr (NTENS == 3)
                    bulk_g2s(stage_ptr(issue_stage, 2), tile_src(in2, row0, l2, off), bytes, bar,
                             policy);
            } else {
                mbar_arrive_expect_tx(bar, (uint32_t)nr * row_bytes * NTENS);
                issue_copies(issued, issue_stage, 0, 1);
            }
        }
        advance();
    };
    // Timeout exit: flag it, then wait (bounded) for this CTA's copies that
    // may still be landing in shared memory before the CTA retires (at most
    // the last S issued tiles: an earlier stage was consumed before it was
    // issued again).
    // Claimed tiles: the last CTA to finish puts the counter back to zero for
    // the next launch handed it, which reads it only once this grid has
    // completed (every CTA counts itself once, after its last claim).
    auto finish_claims = [&]() {
        if (dyn && tid == 0) {
            unsigned long long *done = a.tile_ctr + CLAIM_STRIDE * CLAIM_MAX_K;
            __threadfence();
            if (atomicAdd(done, 1ull) == (unsigned long long)grid - 1ull) {
                __threadfence();
                for (int j = 0; j < CK; ++j) atomicExch(a.tile_ctr + CLAIM_STRIDE * j, 0ull);
                atomicExch(done, 0ull);
            }
        }
    };
    auto fail = [&]() {
        if (tid == 0) {
            atomicOr(a.status, DEVSTATUS_WAIT_TIMEOUT);
            for (int64_t kk = max((int64_t)0, issued - S); kk < issued; ++kk) {
                const int64_t t = dyn ? stage_tile[kk % S] : (int64_t)blockIdx.x + kk * grid;
                if (t == a.drop_tile) continue;
                mbar_wait_bounded(&full[kk % S], (uint32_t)((kk / S) & 1), DEFAULT_WAIT_BUDGET);
            }
        }
        finish_claims();
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Launched as a programmatic dependent: nothing in global memory may be
    // touched before the previous kernel on the stream has completed.
    griddep_wait();
    if (dyn && tid == 0) pending = (int64_t)atomicAdd(c_ctr, 1ull);  // used after the fixed tiles
    {
        const int64_t n0 = dyn ? (int64_t)S : min((int64_t)S, nk);
        if constexpr (SPREAD_COPIES) {
            if (tmap_mode) {
                if (tid == 0)
                    while (issued < n0) issue_tmap();
            } else {
                if (tid == 0)
                    for (int64_t i = 0; i < n0; ++i) post_expect(i, (int)i);
                __syncthreads();  // the expected bytes are posted before any copy
                for (int64_t i = 0; i < n0; ++i) {
                    issue_copies(i, issue_stage, tid, NT);
                    advance();
                }
            }
        } else if (tid == 0) {
            while (issued < n0 && more()) issue_next();
        }
    }

    // w' = weight_bias + w for the columns this thread owns, in fp32.
    float2 wp[V][VP];
    {
        const float2 wb2 = make_float2(a.weight_bias, a.weight_bias);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G;
            float2 wf[VP];
            if constexpr (SH) {
                // this thread's columns: hd + vi * EPV + e (w has its own
                // alignment; read once per CTA, element by element)
                const T *wt = static_cast<const T *>(a.w);
                const int c0 = hd + vi * EPV;
#pragma unroll
                for (int q = 0; q < VP; ++q) {
                    wf[q].x = vi < NB ? Cvt<T>::load1(wt + c0 + 2 * q) : 0.f;
                    wf[q].y = vi < NB ? Cvt<T>::load1(wt + c0 + 2 * q + 1) : 0.f;
                }
            } else {
                const uint4 wv =
                    vi < NV ? reinterpret_cast<const uint4 *>(a.w)[vi] : make_uint4(0, 0, 0, 0);
                unpack_vec<T>(wv, wf);
            }
#pragma unroll
            for (int q = 0; q < VP; ++q) wp[j][q] = f2add(wb2, wf[q]);
        }
    }
    // SH: this lane's edge columns, their w' and (VJP) gw accumulators.
    int ecol[ES];
    float ewp[ES], eacc[ES];
#pragma unroll
    for (int e = 0; e < ES; ++e) {
        ecol[e] = edge_col(e);
        ewp[e] = ecol[e] >= 0 ? a.weight_bias + Cvt<T>::load1(static_cast<const T *>(a.w) + ecol[e])
                              : 0.f;
        eacc[e] = 0.f;
    }
    // Element c of a row whose copy's frame starts at vector pointer r.
    auto row_elem = [&](const uint4 *r, int c) -> float {
        return Cvt<T>::load1(reinterpret_cast<const T *>(reinterpret_cast<const unsigned char *>(r) + shm) + c);
    };
    float2 acc[VJP ? V : 1][VP];
#pragma unroll
    for (int j = 0; j < (VJP ? V : 1); ++j)
#pragma unroll
        for (int q = 0; q < VP; ++q) acc[j][q] = make_float2(0.f, 0.f);

    // Where vector j of a tile's row q sits in the stage: col[j] + q * row_step
    // (general sub-warp instance: column boxes; otherwise plain rows, vi + q * NV).
    int col[SPREAD_COPIES ? V : 1];
    int row_step = NV;
    if constexpr (SPREAD_COPIES) {
        const int bwv = BC / EPV;  // vectors per box row
        row_step = bwv;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G, b = vi / bwv;
            col[j] = b * (TR * bwv) + (vi - b * bwv);
        }
    }

    // One row: load this thread's vectors from the stage into fp32 (h = x +
    // residual, or x; the VJP also g), and its partial sum(h^2) and, for the
    // VJP, partial dot = sum(g * w' * x).
    auto load_row = [&](const uint4 *r0, const uint4 *r1, float2 (&xa)[V][VP],
                        float2 (&xb)[V][VP], float &sa, float &sb) {
        float2 s2 = make_float2(0.f, 0.f), d2 = make_float2(0.f, 0.f);
        if constexpr (SH) {  // this lane's edge elements
#pragma unroll
            for (int e = 0; e < ES; ++e) {
                if (ecol[e] >= 0) {
                    float x = row_elem(r0, ecol[e]);
                    const float y = NTENS >= 2 ? row_elem(r1, ecol[e]) : 0.f;
                    if constexpr (MODE == MODE_FWD_RES) x = x + y;  // h
                    s2.x = fmaf(x, x, s2.x);
                    if constexpr (VJP) d2.x = fmaf(y * ewp[e], x, d2.x);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G;
            if (vi < NB) {
                const int si = SPREAD_COPIES ? col[SPREAD_COPIES ? j : 0] : vi + bo;
                unpack_vec<T>(r0[si], xa[j]);
                if constexpr (NTENS >= 2) unpack_vec<T>(r1[si], xb[j]);
                if constexpr (MODE == MODE_FWD_RES) {
#pragma unroll
                    for (int q = 0; q < VP; ++q) xa[j][q] = f2add(xa[j][q], xb[j][q]);  // h
                }
#pragma unroll
                for (int q = 0; q < VP; ++q) s2 = f2fma(xa[j][q], xa[j][q], s2);
                if constexpr (VJP) {
#pragma unroll
                    for (int q = 0; q < VP; ++q) d2 = f2fma(f2mul(xb[j][q], wp[j][q]), xa[j][q], d2);
                }
            }
        }
        sa = s2.x + s2.y;
        sb = d2.x + d2.y;
    };

    // Outputs of one row from the registers load_row filled (the fused-op VJP
    // also reads its row of the new_residual gradient, r2, from the stage).
    auto row_outputs = [&](const float2 (&xa_in)[V][VP], const float2 (&xb_in)[V][VP],
                           const uint4 *r0, const uint4 *r1, const uint4 *r2, int64_t row, float r,
                           float dot) {
        const size_t base0 = (size_t)(row * lo0), base1 = (size_t)(row * lo1);
        // SH: whole vector vi of a row is vector vi + bo of its output row's
        // aligned frame (the outputs have the inputs' offset)
        uint4 *o0 = out0 + base0, *o1 = out1 + base1;
        if constexpr (SH) {
            o0 = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.out0) + row * row_bytes - shm) + bo;
            if constexpr (MODE == MODE_FWD_RES)
                o1 = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.out1) + row * row_bytes -
                                               shm) + bo;
        }
        auto store_vec = [&](uint4 *orow, int vi, const float2 (&f)[VP]) {
            st_global(orow + vi, pack_vec<T>(f));
        };
        const float2 rr = make_float2(r, r);
        const float c = (r * r) * (dot * inv_D);  // r^2 * dot / D
        const float2 nc2 = make_float2(-c, -c);
        if constexpr (SH) {  // this lane's edge elements, one at a time
            T *orow0 = static_cast<T *>(a.out0) + row * (int64_t)D;
#pragma unroll
            for (int e = 0; e < ES; ++e) {
                if (ecol[e] >= 0) {
                    float x = row_elem(r0, ecol[e]);
                    const float y = NTENS >= 2 ? row_elem(r1, ecol[e]) : 0.f;
                    if constexpr (VJP) {
                        float o = r * (y * ewp[e] - x * c);
                        eacc[e] = fmaf(y, x * r, eacc[e]);
                        if constexpr (ADD) o = o + row_elem(r2, ecol[e]);
                        Cvt<T>::store1(orow0 + ecol[e], o);
                    } else {
                        if constexpr (MODE == MODE_FWD_RES) {
                            x = x + y;
                            Cvt<T>::store1(static_cast<T *>(a.out1) + row * (int64_t)D + ecol[e], x);
                        }
                        Cvt<T>::store1(orow0 + ecol[e], (x * r) * ewp[e]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G;
            if (vi < NB) {
                float2 o[VP];
                const float2 *xa = xa_in[j], *xb = xb_in[j];
                float2 ra[VP], rb[VP];
                if constexpr (RELOAD) {
                    const int si = SPREAD_COPIES ? col[SPREAD_COPIES ? j : 0] : vi + bo;
                    unpack_vec<T>(r0[si], ra);
                    unpack_vec<T>(r1[si], rb);
                    xa = ra;
                    xb = rb;
                }
                if constexpr (VJP) {
#pragma unroll
                    for (int q = 0; q < VP; ++q) {
                        const float2 u = f2mul(xb[q], wp[j][q]);           // g w'
                        o[q] = f2mul(f2fma(xa[q], nc2, u), rr);             // r (g w' - x c)
                        acc[j][q] = f2fma(xb[q], f2mul(xa[q], rr), acc[j][q]);  // g x r
                    }
                    if constexpr (ADD) {
                        float2 gr[VP];
                        unpack_vec<T>(r2[SPREAD_COPIES ? col[SPREAD_COPIES ? j : 0] : vi + bo], gr);
#pragma unroll
                        for (int q = 0; q < VP; ++q) o[q] = f2add(o[q], gr[q]);  // + g_new_residual
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < VP; ++q) o[q] = f2mul(f2mul(xa[q], rr), wp[j][q]);
                    if constexpr (MODE == MODE_FWD_RES) store_vec(o1, vi, xa_in[j]);
                }
                store_vec(o0, vi, o);
            }
        }
    };

    int s = 0;        // stage of tile k
    uint32_t ph = 0;  // parity of that stage's phase
    if constexpr (CTA_ROW) {
        for (int64_t k = 0; dyn || k < nk; ++k) {
            int64_t row = (int64_t)blockIdx.x + k * grid;  // tile_rows == 1
            // The VJP may be handed the forward's scale; fetch it early.
            const float r_saved = (GEN && VJP && a.rstd) ? __ldg(a.rstd + row) : 0.f;
            const bool ok = mbar_wait_bounded(&full[s], ph, a.wait_budget);
            bool end = false;  // claimed tiles: the stage says none is left
            if (dyn) {
                row = ok ? stage_tile[s] : 0;
                end = ok && row < 0;
            }
            float2 xa[V][VP], xb[V][VP];
            float sa, sb;
            load_row(reinterpret_cast<const uint4 *>(stage_ptr(s, 0)),
                     reinterpret_cast<const uint4 *>(stage_ptr(s, NTENS >= 2 ? 1 : 0)), xa, xb, sa,
                     sb);
            sa = group_sum<32>(sa);
            if constexpr (VJP) sb = group_sum<32>(sb);
            float2 *rb = red + (k & 1) * NWARPS;
            if (lane == 0) rb[warp] = make_float2(sa, sb);
            // Everyone has finished row k-1 (its stage is free again) and has
            // published row k's warp totals.
            if (__syncthreads_or(!ok)) {
                fail();
                return;
            }
            if (end) break;  // every thread read the same stage word
            if (tid == 0 && k >= 1 && more()) issue_next();
            // Each group of WP lanes (the warp count rounded up to a power of
            // two) sums all warp totals: the same sums a 32-lane tree with
            // zeros past NWARPS gives, in log2(WP) shuffle levels.
            const int wl = lane & (WP - 1);
            float2 tot = wl < NWARPS ? rb[wl] : make_float2(0.f, 0.f);
            tot.x = group_sum<WP>(tot.x);
            if constexpr (VJP) tot.y = group_sum<WP>(tot.y);
            float r = rsqrtf(tot.x * inv_D + eps);
            if constexpr (GEN && VJP) {
                if (a.rstd) r = r_saved;
            } else if constexpr (GEN) {
                if (a.rstd && tid == 0) a.rstd[row] = r;
            }
            row_outputs(xa, xb, reinterpret_cast<const uint4 *>(stage_ptr(s, 0)),
                        reinterpret_cast<const uint4 *>(stage_ptr(s, NTENS >= 2 ? 1 : 0)),
                        reinterpret_cast<const uint4 *>(stage_ptr(s, NTENS - 1)), row, r,
                        tot.y);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else {
        for (int64_t k = 0; dyn || k < nk; ++k) {
            int64_t row0 = ((int64_t)blockIdx.x + k * grid) * TR;
            int nr = (int)min((int64_t)TR, rows - row0);
            // The VJP may be handed the forward's scale: fetch this thread's
            // first row's early, and each next row's one row ahead.
            float r_next = 0.f;
            if constexpr (GEN && VJP)
                if (a.rstd && gid < nr) r_next = __ldg(a.rstd + row0 + gid);
            const bool ok = mbar_wait_bounded(&full[s], ph, a.wait_budget);
            bool end = false;  // claimed tiles: the stage says none is left
            if (dyn) {
                const int64_t t = ok ? stage_tile[s] : -1;
                end = ok && t < 0;
                row0 = t < 0 ? 0 : t * TR;
                nr = t < 0 ? 0 : (int)min((int64_t)TR, rows - row0);
            }
            const uint4 *t0 = reinterpret_cast<const uint4 *>(stage_ptr(s, 0));
            const uint4 *t1 = reinterpret_cast<const uint4 *>(stage_ptr(s, NTENS >= 2 ? 1 : 0));
            const uint4 *t2 = reinterpret_cast<const uint4 *>(stage_ptr(s, NTENS - 1));
            // Row q of the tile in the stage: q * row_step vectors in (SH: the
            // aligned vector holding its first byte; the tile's copy starts at
            // the aligned boundary below its first row)
            const uint32_t toff = tile_off(row0);
            auto rstep = [&](int q) -> size_t {
                return SH ? (size_t)((toff + (uint32_t)q * row_bytes) >> 4) : (size_t)q * row_step;
            };
            for (int qb = 0; qb < TR; qb += NG) {  // same trip count in every lane
                const int q = qb + gid;
                const bool valid = q < nr;
                const float r_saved = r_next;
                if constexpr (GEN && VJP)
                    if (a.rstd && q + NG < nr) r_next = __ldg(a.rstd + row0 + q + NG);
                float2 xa[V][VP], xb[V][VP];
                float sa = 0.f, sb = 0.f;
                if (valid) load_row(t0 + rstep(q), t1 + rstep(q), xa, xb, sa, sb);
                sa = group_sum<G>(sa);
                if constexpr (VJP) sb = group_sum<G>(sb);
                if (valid && ok) {
                    float r = rsqrtf(sa * inv_D + eps);
                    if constexpr (GEN && VJP) {
                        if (a.rstd) r = r_saved;
                    } else if constexpr (GEN) {
                        if (a.rstd && gl == 0) a.rstd[row0 + q] = r;
                    }
                    row_outputs(xa, xb, t0 + rstep(q), t1 + rstep(q), t2 + rstep(q), row0 + q, r, sb);
                }
            }
            // Thread 0 has seen the stage's phase complete (ok), so the next
            // phase may take its expected bytes now.
            if constexpr (SPREAD_COPIES)
                if (!tmap_mode && tid == 0 && ok && issued < nk) post_expect(issued, issue_stage);
            if (__syncthreads_or(!ok)) {  // the whole tile is consumed
                fail();
                return;
            }
            if (end) break;  // every thread read the same stage word
            if constexpr (SPREAD_COPIES) {
                if (tmap_mode) {
                    if (tid == 0 && issued < nk) issue_tmap();
                } else if (issued < nk) {
                    issue_copies(issued, issue_stage, tid, NT);
                    advance();
                }
            } else if (tid == 0 && more()) {
                issue_next();
            }
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    }

    finish_claims();
    // The next kernel on the stream may start launching (it waits for this
    // one to complete before touching memory).
    griddep_launch_dependents();
    if constexpr (VJP) {
        float *prow = a.partials + (size_t)blockIdx.x * D;
        // EPV consecutive fp32 columns of one vector's accumulators.
        auto store_acc = [&](float *dst, int j) {
#pragma unroll
            for (int u = 0; u < VP / 2; ++u)
                reinterpret_cast<float4 *>(dst)[u] =
                    make_float4(acc[j][2 * u].x, acc[j][2 * u].y, acc[j][2 * u + 1].x, acc[j][2 * u + 1].y);
        };
        // SH: this thread's columns of vector j start at hd + vi * EPV (stored
        // one by one), its edge columns at ecol[].
        auto store_acc_sh = [&](float *dst_row, int j, int vi) {
            const int c0 = hd + vi * EPV;
#pragma unroll
            for (int q = 0; q < VP; ++q) {
                dst_row[c0 + 2 * q] = acc[j][q].x;
                dst_row[c0 + 2 * q + 1] = acc[j][q].y;
            }
        };
        auto store_edge_acc = [&](float *dst_row) {
#pragma unroll
            for (int e = 0; e < ES; ++e)
                if (ecol[e] >= 0) dst_row[ecol[e]] = eacc[e];
        };
        if constexpr (CTA_ROW) {
            // Each column is owned by exactly one thread of the CTA.
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = gl + j * G;
                if constexpr (SH) {
                    if (vi < NB) store_acc_sh(prow, j, vi);
                } else {
                    if (vi < NV) store_acc(prow + (size_t)vi * EPV, j);
                }
            }
            if constexpr (SH) store_edge_acc(prow);
        } else {
            // NG groups own the same columns: add their registers in group
            // order through shared memory (the ring is idle now).
            __syncthreads();
            float *buf = reinterpret_cast<float *>(ring);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = gl + j * G;
                if constexpr (SH) {
                    if (vi < NB) store_acc_sh(buf + (size_t)gid * D, j, vi);
                } else {
                    if (vi < NV) store_acc(buf + (size_t)gid * D + (size_t)vi * EPV, j);
                }
            }
            if constexpr (SH) store_edge_acc(buf + (size_t)gid * D);
            __syncthreads();
            for (int col = tid; col < D; col += NT) {
                float sum = 0.f;
                for (int gg = 0; gg < NG; ++gg) sum += buf[(size_t)gg * D + col];
                prow[col] = sum;
            }
        }
    }
}

}  // namespace rmsn
