/*
 * rmsnorm.h -- C ABI of librmsnorm_gb300.so: the row-wise RMSNorm hot path on
 * one GB300 (sm_103a).  Plain pointers and sizes only; no C++ or framework
 * types cross this boundary.
 *
 * Operations (sources are web pages, named by title and section):
 *
 *   rmsnorm_fwd -- fused residual-add RMSNorm forward, two outputs.
 *     "Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
 *     Background, FusedAddRMSNorm bullet: h = x + residual, then
 *     out = h * rsqrt(mean(h^2) + eps) * (weight_bias + w) in one pass, the fp32
 *     sum kept once, a warp-then-block sum of squares; weight_bias = 1 gives the
 *     Gemma (1 + w) convention.  Same page, Background, last paragraph: the
 *     residual update is a second output (normed, new_residual).
 *
 *   rmsnorm_vjp -- RMSNorm VJP: gx and a gw reduced across rows on the GPU.
 *     "RMSNormVJP backward writes a full {n_rows, D} gw_temp intermediate",
 *     Proposed changes: gw must not go through a {n_rows, D} temporary that a
 *     second kernel re-reduces; rows are combined inside the kernel.  POC: the
 *     gradients of sum(rms_norm(x, w, eps) * y) with respect to x and w.
 *
 * Definitions, per row of D elements (h = x + residual, or x):
 *     ms = (1/D) sum_j h_j^2,  r = 1 / sqrt(ms + eps),  w'_j = weight_bias + w_j
 *     out_j = h_j * r * w'_j,   new_residual_j = h_j
 *     dot = sum_j g_j * w'_j * h_j
 *     gx_j = r * g_j * w'_j - (r^3 / D) * h_j * dot
 *     gw_j = sum over rows of g_j * h_j * r
 *
 * Numerics: inputs and outputs are fp16, bf16 or fp32; all arithmetic is fp32;
 * every fp16/bf16 output element is rounded once, to nearest-even, from fp32.
 * h is normalised unrounded (the fp32 sum), new_residual is its rounding.  gw
 * is fp32 and bit-identical from run to run on the same device for the same
 * (rows, D, dtype, strides): its summation order is fixed and does not depend
 * on timing.
 *
 * Layout and ownership: every tensor is a row-major device buffer owned by the
 * caller: x, residual, out, new_residual, g, gx are [rows, D] of dtype, dense
 * (rows D elements apart) for rmsnorm_fwd / rmsnorm_vjp / rmsnorm_fused_vjp,
 * or with a row stride of their own (>= D elements; elements of a row are
 * contiguous) for rmsnorm_fwd_ex / rmsnorm_vjp_ex; w is [D] of dtype, dense;
 * gw and rstd are fp32, dense.  Pointers must be device pointers of the
 * current device (cudaGetDevice) and `stream` a cudaStream_t of that device
 * (NULL = legacy default stream), passed as void*.  Any alignment is accepted;
 * 16-byte aligned pointers and row strides with D * sizeof(element) a
 * multiple of 16 take the fast kernels.
 *
 * Aliasing: an output may be the very same tensor as an input (same pointer
 * and row stride: out == x, new_residual == residual, gx == g, ...): every
 * element is read before the same thread writes it.  Any other overlap, and
 * any overlap of two outputs, is rejected with RMSNORM_ERR_INVALID_ARG.  For
 * tensors with equal row strides the test is exact, so the disjoint halves of
 * one [rows, 2D] buffer are accepted as two tensors of row stride 2D; tensors
 * with different strides must not share their address ranges.
 *
 * Asynchrony and errors: calls enqueue work on `stream` and return without
 * synchronising.  Every call returns an rmsnorm_status_t and never aborts.
 * Host-side validation fails before anything is enqueued.  A CUDA error at
 * launch gives RMSNORM_ERR_CUDA; rmsnorm_last_cuda_error() then returns the
 * cudaError_t of the calling thread's last failure.  A kernel whose bounded
 * wait for its own asynchronous copies runs out (about a second) stops, leaves
 * its outputs undefined and sets RMSNORM_DEVSTATUS_WAIT_TIMEOUT in the
 * library's device status word, read by rmsnorm_device_status().
 *
 * Row scheduling of the forward: the CTAs of the staged forward kernels take
 * most of their rows from counters at run time, so a CTA the memory system
 * slows down takes fewer; the results do not depend on which CTA takes a row.
 * The counters are sets in the library's device memory that every launch
 * leaves at zero.  Launches outside a graph capture take them in turn from
 * 16384 sets; a launch recorded into a graph keeps a set of its own, which
 * every replay of that graph instance uses (a graph instance never runs
 * alongside itself).  Two instances made from one captured graph must
 * therefore not run at the same time; the environment setting
 * RMSNORM_TUNE=claim=0, read once per process, turns the counters off (the
 * CTAs then take fixed rows).
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RMSNORM_F16 = 0,  /* IEEE binary16 */
    RMSNORM_BF16 = 1, /* bfloat16 */
    RMSNORM_F32 = 2   /* IEEE binary32 (norm entry points only; the gate and
                         the rotary embedding take fp16 or bf16) */
} rmsnorm_dtype_t;

typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_INVALID_ARG = 1,  /* null pointer, D <= 0, rows < 0, bad dtype,
                                     eps < 0 or not finite, weight_bias not
                                     finite, residual/new_residual mismatch,
                                     row stride < D, overlapping buffers, too
                                     small workspace */
    RMSNORM_ERR_UNSUPPORTED = 2,  /* D > RMSNORM_MAX_D, or rows * D overflows */
    RMSNORM_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    RMSNORM_ERR_NO_MEMORY = 4,    /* scratch allocation failed */
    RMSNORM_ERR_TIMEOUT = 5       /* a device-side bounded wait ran out */
} rmsnorm_status_t;

/* Largest supported row length. */
#define RMSNORM_MAX_D ((int64_t)1 << 24)

/* Bits of the device status word. */
#define RMSNORM_DEVSTATUS_WAIT_TIMEOUT 1u
#define RMSNORM_DEVSTATUS_BAD_INDEX 2u /* rmsnorm_rope_kv_append: a position or
                                          slot out of range (that token skipped) */

/*
 * Fused residual-add RMSNorm forward.
 *   x            [rows, D] dtype, input.
 *   residual     [rows, D] dtype, or NULL for plain RMSNorm (h = x).
 *   w            [D] dtype, weight.
 *   eps          >= 0, added to the mean square inside the root.
 *   weight_bias  scalar added to every w_j in fp32 (0: standard, 1: Gemma).
 *   out          [rows, D] dtype, normalised output.
 *   new_residual [rows, D] dtype, receives round(x + residual); must be NULL
 *                exactly when residual is NULL.
 * rows == 0 is a no-op returning RMSNORM_OK.
 */
int rmsnorm_fwd(const void *x, const void *residual, const void *w, float eps,
                float weight_bias, void *out, void *new_residual, int64_t rows,
                int64_t D, int dtype, void *stream);

/*
 * RMSNorm VJP.
 *   x   [rows, D] dtype, the tensor that was normalised (for the fused
 *       forward pass its new_residual; the gradient with respect to both x and
 *       residual of the fused op is then gx plus whatever gradient reaches
 *       new_residual, which the caller adds).
 *   w   [D] dtype;  g [rows, D] dtype, the incoming gradient of out.
 *   gx  [rows, D] dtype, gradient with respect to x.
 *   gw  [D] fp32, gradient with respect to w, summed over rows; overwritten
 *       (rows == 0 writes zeros).
 * The per-CTA gw partials ([P, D] fp32 with P about the SM count) live in
 * scratch that this call takes and returns stream-ordered on `stream` from a
 * memory pool the library keeps per device (cudaMallocFromPoolAsync /
 * cudaFreeAsync; the pool holds on to freed memory for the next call);
 * allocation failure returns RMSNORM_ERR_NO_MEMORY.  No [rows, D] temporary
 * is ever allocated.  A call that runs as a single CTA (one row) writes its one
 * partial row straight into gw when gw is 16-byte aligned: no scratch, one
 * kernel, the same bits.  A decode-sized call of 2-8 rows (16-byte aligned
 * rows of up to 2048 vectors) runs as one thread-block cluster of its rows
 * that adds the rows' contributions in row order itself and, with gw 16-byte
 * aligned, writes gw directly: no scratch, one kernel.
 */
int rmsnorm_vjp(const void *x, const void *w, const void *g, float eps,
                float weight_bias, void *gx, float *gw, int64_t rows, int64_t D,
                int dtype, void *stream);

/*
 * VJP of the two-output fused op (out, new_residual) = fused forward of
 * (x, residual, w).  Source: "Fused residual-add RMSNorm and fused RoPE +
 * KV-append decode kernels", Background: the residual update is a second
 * output, so a gradient can reach it as well as out.
 *   h           [rows, D] dtype, the new_residual the forward produced.
 *   g_out       [rows, D] dtype, the gradient of out.
 *   g_residual  [rows, D] dtype, the gradient of new_residual, or NULL (none).
 *   g_h         [rows, D] dtype, receives VJP(h, g_out) + g_residual, rounded
 *               once: the gradient with respect to x and to residual alike.
 *   gw          [D] fp32, as for rmsnorm_vjp (new_residual does not depend on w).
 * One pass over h, g_out and g_residual; scratch, errors and aliasing (g_h may
 * be g_out or g_residual) as for rmsnorm_vjp.  With g_residual == NULL this is
 * rmsnorm_vjp.
 */
int rmsnorm_fused_vjp(const void *h, const void *w, const void *g_out,
                      const void *g_residual, float eps, float weight_bias, void *g_h,
                      float *gw, int64_t rows, int64_t D, int dtype, void *stream);

/*
 * The forward with row strides and the per-row scale.  As rmsnorm_fwd, plus:
 *   ld_x, ld_residual, ld_out, ld_new_residual  row strides in elements
 *                (>= D; ignored for a NULL tensor and when rows == 1).
 *   rstd         [rows] fp32, receives r_i = 1 / sqrt(mean(h_i^2) + eps), the
 *                value row i was multiplied by, for reuse by rmsnorm_vjp_ex;
 *                or NULL.
 * Sources: the forward's definition above (the rsqrt factor of the
 * FusedAddRMSNorm bullet); the pages do not name strided rows or a saved
 * rstd: they are the layout of a slice of a wider buffer and the scalar a
 * backward pass would otherwise recompute.  rmsnorm_fwd is this call with
 * every stride D and rstd NULL.
 */
int rmsnorm_fwd_ex(const void *x, int64_t ld_x, const void *residual, int64_t ld_residual,
                   const void *w, float eps, float weight_bias, void *out, int64_t ld_out,
                   void *new_residual, int64_t ld_new_residual, float *rstd, int64_t rows,
                   int64_t D, int dtype, void *stream);

/*
 * The VJP (plain, or of the two-output fused op) with row strides and an
 * optional saved per-row scale.  As rmsnorm_fused_vjp (g_residual NULL gives
 * rmsnorm_vjp), plus:
 *   ld_x, ld_g, ld_g_residual, ld_gx  row strides in elements (>= D).
 *   rstd   [rows] fp32 or NULL.  Given, row i uses r = rstd[i] in place of
 *          1 / sqrt(mean(x_i^2) + eps) (eps is then unused); pass what
 *          rmsnorm_fwd_ex wrote for the same rows.  It saves the sum of
 *          squares (arithmetic only: the same bytes move either way).
 * gw scratch comes from the library's pool as for rmsnorm_vjp.
 */
int rmsnorm_vjp_ex(const void *x, int64_t ld_x, const void *w, const void *g, int64_t ld_g,
                   const void *g_residual, int64_t ld_g_residual, const float *rstd, float eps,
                   float weight_bias, void *gx, int64_t ld_gx, float *gw, int64_t rows, int64_t D,
                   int dtype, void *stream);

/*
 * Bytes of scratch rmsnorm_vjp_ws needs for this problem on the current
 * device (0 when rows == 0).  Returns 0 for invalid arguments as well.
 */
size_t rmsnorm_vjp_workspace_size(int64_t rows, int64_t D, int dtype);

/*
 * rmsnorm_vjp with caller-owned scratch: `workspace` is a device buffer of at
 * least rmsnorm_vjp_workspace_size(rows, D, dtype) bytes, 256-byte aligned.
 * Its contents on entry do not matter; it must not be used by other work while
 * this call runs on `stream`.
 */
int rmsnorm_vjp_ws(const void *x, const void *w, const void *g, float eps,
                   float weight_bias, void *gx, float *gw, int64_t rows,
                   int64_t D, int dtype, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * Gated activation of the decode loop.  Source: "Fused residual-add RMSNorm
 * and fused RoPE + KV-append decode kernels", Background, third bullet (a
 * fused silu(x[:d]) * x[d:2d] gate with 16-byte vectorised loads).
 *   x    [rows, 2*d] dtype: each row is [a | b], a and b of d values.
 *   out  [rows, d] dtype: out_j = silu(a_j) * b_j, silu(a) = a / (1 + e^-a),
 *        computed in fp32 and rounded once.
 * out must not overlap x.  d % 8 == 0 with 16-byte aligned pointers takes the
 * vectorised kernel; other shapes and alignments are accepted.  rows == 0 is a
 * no-op.  Errors as for rmsnorm_fwd.
 */
int rmsnorm_gated_silu(const void *x, void *out, int64_t rows, int64_t d, int dtype,
                       void *stream);

/*
 * Rotary embedding of q and k fused with the KV-cache append.  Source: "Fused
 * residual-add RMSNorm and fused RoPE + KV-append decode kernels", Background,
 * second bullet, and Task item 3 (rope on q and k, k and v written into the
 * cache slab or a paged pool block in the same kernel; cos/sin from a
 * precomputed cache or computed on the fly).
 *   q        [T, Hq, Dh] dtype;  q_out [T, Hq, Dh] dtype (may be q: in place).
 *   k, v     [T, Hkv, Dh] dtype.
 *   positions, slots  [T] int64, device memory: token t's absolute position
 *            and the cache row it goes to (negative: not written).  A dense
 *            slab uses slot = position (a ring / sliding window: position mod
 *            window); a paged pool [blocks, block_size, Hkv, Dh] uses
 *            slot = block * block_size + offset.
 *   k_cache, v_cache  [num_slots, Hkv, Dh] dtype: row slots[t] receives the
 *            rotated k and the v of token t; other rows are untouched.
 *   cos_sin  [max_pos, Dh] fp32 device table (Dh/2 cosines then Dh/2 sines of
 *            each position), or NULL: theta_i = position * rope_base^(-2i/Dh)
 *            computed on the fly (about 1e-8 rad of error up to 1e6).
 *   interleaved  0: pairs (i, i + Dh/2) (rotate-half); 1: pairs (2i, 2i + 1).
 * Arithmetic in fp32, each output rounded once.  Dh even, at most 1024;
 * Dh % 16 == 0 with 16-byte aligned pointers takes the vectorised kernel.
 * Positions outside [0, max_pos) (or negative) and slots >= num_slots are
 * detected on the device: the token's outputs are skipped (nothing out of
 * range is touched) and RMSNORM_DEVSTATUS_BAD_INDEX is set.  The caches must
 * not overlap each other, the inputs or q_out.  T == 0 is a no-op.
 * (rmsnorm_ is this library's symbol prefix.)
 */
int rmsnorm_rope_kv_append(const void *q, const void *k, const void *v,
                           const int64_t *positions, const int64_t *slots, void *q_out,
                           void *k_cache, void *v_cache, const float *cos_sin,
                           int64_t max_pos, float rope_base, int interleaved, int64_t T,
                           int64_t Hq, int64_t Hkv, int64_t Dh, int64_t num_slots, int dtype,
                           void *stream);

/* Size of the fixed device array behind rmsnorm_vjp_noalloc: 16 MiB. */
#define RMSNORM_VJP_NOALLOC_MAX_BYTES ((size_t)16 << 20)

/*
 * rmsnorm_vjp for callers that cannot allocate device memory.  The pages
 * have no counterpart: this entry point exists for programs that may not call
 * cudaMalloc or any other allocator when they run the backward pass (runtimes
 * that reserve all device memory at start-up and forbid later allocations,
 * plugin interfaces that give a kernel neither an allocator nor a workspace,
 * latency-critical loops that cannot afford an allocation's synchronisation
 * or its failure).  Arguments, results, numerics and errors are those of
 * rmsnorm_vjp; the gw partial rows go to a 16 MiB array compiled into the
 * library instead of allocated memory, and nothing is allocated.
 *   - Memory: the array occupies RMSNORM_VJP_NOALLOC_MAX_BYTES of device memory
 *     on every GPU where the library is loaded, until the process exits.
 *   - Limit: a problem whose scratch (one fp32 row of D per partial row of
 *     the plan these pointers get) exceeds RMSNORM_VJP_NOALLOC_MAX_BYTES
 *     returns RMSNORM_ERR_UNSUPPORTED and enqueues nothing.  On a 152-SM
 *     GB300, at any row count: dense fp16/bf16 rows up to D = 131072 and fp32
 *     rows up to D = 65536 whose tensors start on 16-byte boundaries (one
 *     partial row per CTA of the CTA-per-row and sub-warp tiers, one per
 *     cluster of the cluster tier: at most 10 MB), and dense rows whose
 *     tensors all start at one shared offset from a boundary up to D = 16383
 *     (fp16/bf16) or 8191 (fp32).  Anything else (tensors at different offsets, strided rows off
 *     boundaries, longer rows) runs on the element-at-a-time tier with
 *     max(min(rows, 8), min(2 x SMs, rows * 3 * size / 40)) partial rows,
 *     which fit while that count x D x 4 bytes <= 16 MiB (e.g. D <= 13,797
 *     at 2,000 or more rows).
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, and it keeps the
 *     last call's contents (nothing in it needs to start at zero: each call
 *     writes every partial row before reading it).  Calls whose work overlaps
 *     on the GPU (other streams, or other host threads) race on the array and
 *     give wrong gw; order them on one stream.
 */
int rmsnorm_vjp_noalloc(const void *x, const void *w, const void *g, float eps,
                        float weight_bias, void *gx, float *gw, int64_t rows,
                        int64_t D, int dtype, void *stream);

/* Static, human-readable name of a status code. */
const char *rmsnorm_status_string(int status);

/* cudaError_t of the calling thread's last RMSNORM_ERR_CUDA (0 if none). */
int rmsnorm_last_cuda_error(void);

/*
 * Reads the device status word of the current device into *bits (a mask of
 * RMSNORM_DEVSTATUS_* flags set by kernels since the last clear) and clears it
 * when `clear` is non-zero.  Synchronises the device: diagnostics only.
 * Returns RMSNORM_ERR_TIMEOUT when the timeout bit is set, else
 * RMSNORM_ERR_INVALID_ARG when the bad-index bit is set.
 */
int rmsnorm_device_status(unsigned int *bits, int clear);

/*
 * Test hook for the timeout path.  Until reset with (-1, 0), the staged
 * kernels launched by the calling process skip the asynchronous copy of the
 * tile with index `drop_tile` (so its wait can never finish) and give every
 * wait `budget_cycles` SM clock cycles instead of the default.  The kernel then
 * reports RMSNORM_DEVSTATUS_WAIT_TIMEOUT, drains its other copies and exits;
 * no fault, trap or hang.  budget_cycles <= 0 restores the default budget.
 */
int rmsnorm_debug_inject(int64_t drop_tile, int64_t budget_cycles);

/*
 * Test hook for the allocation-failure path.  The next `count` gw scratch
 * allocations of rmsnorm_vjp, rmsnorm_fused_vjp and rmsnorm_vjp_ex in this
 * process report failure without calling the allocator: each such call returns
 * RMSNORM_ERR_NO_MEMORY after its argument checks and enqueues nothing (gx and
 * gw are left untouched).  Calls that need no scratch (a VJP that runs as one
 * CTA, rows == 0) and the caller-scratch entry points are not affected and do
 * not use up the count.  count == 0 cancels what is pending; count < 0 returns
 * RMSNORM_ERR_INVALID_ARG.  Host-side only: nothing faults on the device.
 */
int rmsnorm_debug_fail_allocs(int count);

/*
 * Test hook for the staged forwards that take their tiles from counters at
 * run time.  Launches made outside a graph capture normally cycle through
 * 16384 counter sets; after this call they cycle through the first `count`
 * (1 <= count <= 16384), so with count = 1 consecutive forwards reuse one
 * set, which shows that every launch -- one that timed out included --
 * leaves its set at zero.  Forwards that may run at the same time (other
 * streams) must not be launched while count is small.  count == 0 restores
 * the default; other values return RMSNORM_ERR_INVALID_ARG.
 */
int rmsnorm_debug_claim_counters(int count);

/*
 * Describes the kernel plan rmsnorm_fwd (op = 0) or rmsnorm_vjp (op = 1;
 * with has_residual, rmsnorm_fused_vjp with a g_residual) would use for this
 * problem on the current device, as a static string such as
 * "staged:cfg8:nt512:g512:v2:s6:tr1:grid152:smem...:cl0" ("staged-shift:..."
 * for the shifted-rows instances; ":claim" at the end when the CTAs take their
 * rows from counters at run time); for tests and benchmarks.  aligned: 1 = dense
 * tensors at 16-byte aligned addresses (rows off 16-byte boundaries when
 * D * size is not a multiple of 16), 2 = dense tensors that all start at the
 * same unaligned offset, 0 = anything else (strided or mixed offsets).
 */
const char *rmsnorm_describe_dispatch(int op, int64_t rows, int64_t D, int dtype,
                                      int has_residual, int aligned);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
