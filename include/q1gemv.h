/*
 * q1gemv.h -- C ABI of the GB300 Q1_0 (1-bit) GEMV library (libq1gemv.so).
 *
 * The library computes the row-parallel product of 1-bit Q1_0 weights with a
 * q8_0-quantized activation, as bankML's "docs/modules/gpu.md" defines it
 * ("kernels.rs -- the Q1_0 kernels", first bullet):
 *
 *   for every output row, lanes l = 0..7 keep an f32 accumulator a_l = +0;
 *   for every 128-weight block b (in order), with weight scale d0 (fp16):
 *     for every 32-element sub-block k = 0..3, with activation scale d1 (fp16):
 *       s = sum over the lane's 4 elements 32k+4l+i of (bit ? q : -q),
 *           an exact integer, where negating -128 gives -128;
 *       ab = d1*s (k = 0), ab = fma(d1, s, ab) (k = 1..3);
 *     a_l = fma(d0, ab, a_l);
 *   out = ((a0+a4) + (a2+a6)) + ((a1+a5) + (a3+a7)).
 *
 * Every output element equals, bit for bit, the plain CPU definition above on
 * any GPU, launch shape or batch size.
 *
 * Conventions for every call:
 *   - n (activation length) is a multiple of 128, 128 <= n <= 1<<24; rows >= 1,
 *     rows <= 1<<26.
 *   - Pointers are DEVICE pointers owned by the caller unless noted; the
 *     library keeps no reference to them after the call returns.  Buffers must
 *     be 16-byte aligned and must not overlap.  The activation and output
 *     pointers of the products (x, q, d, out) may instead point into pinned
 *     host memory (cudaHostAlloc / cudaHostRegister) where the device can
 *     address it (unified addressing; on a GB300 the kernels then read and
 *     write it over NVLink-C2C, so a host round trip needs no separate copy).
 *     Packed weights must be device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work; nothing blocks the host unless noted.
 *   - Return value: Q1_OK (0) on success, a negative Q1_ERR_* code on a
 *     rejected argument or a CUDA error (nothing is enqueued after a rejected
 *     argument); q1_last_error() then names the call and the reason.
 *   - Activation scales must be finite.  With a non-finite activation scale
 *     the affected outputs are unspecified (never a fault).  Weight scales
 *     must be finite too: q1_0_pack and q2_0_pack reject a block whose fp16
 *     scale is Inf or NaN (Q1_ERR_ARG naming its row and block).
 */
#ifndef Q1GEMV_H
#define Q1GEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q1_OK 0
#define Q1_ERR_ARG (-1)     /* shape, pointer, alignment or size rejected   */
#define Q1_ERR_CUDA (-2)    /* a CUDA runtime call or launch failed         */
#define Q1_ERR_NOMEM (-3)   /* q1_0_verify could not allocate device memory */
#define Q1_MISMATCH 2       /* q1_0_verify: some output differs             */

/* Text of the last error on the calling thread ("" if none).  The pointer is
 * valid until the next library call on the same thread. */
const char *q1_last_error(void);

/* Bytes of the packed weight buffer q1_0_pack writes for a rows x n matrix
 * (18 bytes per 128 weights, rows padded to a multiple of 256 and blocks per
 * row to a multiple of 4).  Returns a negative Q1_ERR_ARG for a bad shape.
 * Host-only; touches no device. */
int64_t q1_0_packed_bytes(int64_t rows, int64_t n);

/* Repack Q1_0 weights once into the library's device layout
 * ("kernels.rs -- the Q1_0 kernels", pack_q1_0 bullet: repacked once, the
 * numbers unchanged, only aligned).
 *   blocks : device, rows*(n/128) consecutive 18-byte blocks, row-major; each
 *            block = fp16 scale d0 (little-endian) + 16 bytes of sign bits,
 *            element j in byte 2 + j/8, bit j%8, 1 = +d0, 0 = -d0.
 *            Only 2-byte alignment is required for this pointer.
 *   packed : device, q1_0_packed_bytes(rows, n) bytes, written entirely.
 * Synchronous: returns after `stream` has finished the packing (see q1_0_gemv).
 * Errors: Q1_ERR_ARG for a bad shape or pointer, or when some block's fp16
 * scale is Inf or NaN (the message names the first such row and block; the
 * packed buffer must then not be used); Q1_ERR_CUDA on a failed launch or
 * copy.  The check uses a few bytes of device memory allocated on `stream`
 * for this call alone, so concurrent calls on other streams or threads do not
 * interfere. */
int q1_0_pack(const uint8_t *blocks, int64_t rows, int64_t n, void *packed, void *stream);

/* Inverse of q1_0_pack: writes rows*(n/128) 18-byte blocks identical to the
 * ones that were packed.  Same pointer rules as q1_0_pack. */
int q1_0_unpack(const void *packed, int64_t rows, int64_t n, uint8_t *blocks, void *stream);

/* q8_0 activation quantization (the q8_0 activation of "kernels.rs", pack_act
 * bullet; scale = max|x| / 127).  For each vector v < nvec and each 32-value
 * block: amax = max|x|, d = amax/127 (f32), id = d ? 1/d : 0 (f32),
 * q = roundf(x*id) (half away from zero), scale stored as fp16 (round to
 * nearest even) of d.
 *   x : device f32 [nvec][n]; q : device int8 [nvec][n];
 *   d : device fp16 bits [nvec][n/32].  Each of the three may instead be
 *   pinned host memory, under the same rule as the products' activations
 *   (one launch then reads x over the host link, in full 512-byte requests).
 * n is a multiple of 32 here (128 for use with the products), 1 <= nvec <= 65535.
 * Inputs must be finite and max|x| <= 65504*127 for the scale to stay finite. */
int q8_quantize_act(const float *x, int64_t nvec, int64_t n, int8_t *q, uint16_t *d, void *stream);

/* Matrix-vector product ("kernels.rs -- the Q1_0 kernels", first and second
 * bullets: one exact dot product per output row; rows are independent).
 *   packed : device, from q1_0_pack(rows, n).
 *   q, d   : device q8_0 activation: int8 [n], fp16 bits [n/32] (any quants,
 *            including -128).
 *   out    : device f32 [rows].
 * Launch uses programmatic dependent launch: the kernel starts streaming
 * `packed` while the preceding kernel on `stream` is still running, and reads
 * q and d only after that kernel's writes are visible.  So `packed` must not be
 * written by the kernel immediately preceding this call on the stream
 * (q1_0_pack and host copies are always complete before it). */
int q1_0_gemv(const void *packed, int64_t rows, int64_t n, const int8_t *q, const uint16_t *d,
              float *out, void *stream);

/* One product of a multi-product call: out = the matrix-vector product of the
 * packed rows x n matrix with one activation vector. */
typedef struct q1_product {
  const void *packed;     /* device, from q1_0_pack(rows, n)                         */
  int64_t rows, n;        /* matrix shape                                            */
  const float *x;         /* device f32 [n]: activation, quantized inside the kernel
                             exactly as q8_quantize_act would; or NULL              */
  const int8_t *q;        /* used when x is NULL: device int8 [n] q8_0 quants        */
  const uint16_t *d;      /* used when x is NULL: device fp16 bits [n/32] scales    */
  float *out;             /* device f32 [rows]                                       */
} q1_product;

#define Q1_MAX_PRODUCTS 256

/* Several independent matrix-vector products in ONE launch (the pages' own
 * next step, "batched submissions ... one wait per group" in "Advantages and
 * efficiency"; e.g. the q/k/v or gate/up products of a layer, or a whole set of
 * independent products).  Each out_j is bit-identical to q8_quantize_act(x_j)
 * (when x_j is given) followed by q1_0_gemv.  Products may differ in shape.
 *   products : HOST array of `count` descriptors (1 <= count <= Q1_MAX_PRODUCTS),
 *              read during the call only.
 * Outputs must not overlap each other or any input.  Same launch behaviour as
 * q1_0_gemv (programmatic dependent launch; `packed` may be read before the
 * preceding kernel on `stream` has finished). */
int q1_0_gemv_multi(const q1_product *products, int count, void *stream);

/* A device byte range (for q1_0_gemv_multi_prefetch). */
typedef struct q1_range {
  const void *ptr;        /* device pointer, 16-byte aligned; NULL with 0 bytes   */
  int64_t bytes;          /* 0 <= bytes <= 2^40, rounded down to a multiple of 16 */
} q1_range;

#define Q1_MAX_PREFETCH_RANGES 4

/* q1_0_gemv_multi, and while the launch runs its CTAs also pull the given
 * device byte ranges into the L2 cache (one bulk prefetch a CTA and range,
 * issued before the kernel waits for the preceding one; nothing waits for
 * them and nothing of them is read into the SMs).  For a chain of dependent
 * launches (a decode step, where each product's activation is produced by the
 * kernels before it), the ranges are the packed weights of the launch that
 * follows (they do not depend on the chain) and its activation (in a decode
 * step the output of the kernel just before, already in L2; a chain that
 * reads stored activations gets the same effect by prefetching them).  That
 * launch then finds its inputs in L2 instead of HBM.  A prefetch never
 * changes what a kernel reads: L2 is where every write lands first.  No
 * counterpart in the pages; it serves their point that each matrix call pays
 * its own submit and wait ("Limitations").
 *   prefetch : HOST array of `nranges` ranges (0 <= nranges <=
 *              Q1_MAX_PREFETCH_RANGES; NULL with 0), read during the call
 *              only.  Each range must be memory the device may read; its
 *              contents do not matter and no byte outside it is touched.
 * Outputs are those of q1_0_gemv_multi, bit for bit.  Q1_ERR_ARG for a bad
 * range, as for the products. */
int q1_0_gemv_multi_prefetch(const q1_product *products, int count, const q1_range *prefetch, int nranges,
                             void *stream);

/* The work split of a q1_0_gemv_multi launch, as the call would make it.
 * Planning only: nothing is launched and no pointer in `products` is read
 * (only rows and n; the shapes are checked as q1_0_gemv_multi checks them).
 * A tile is rows_per_thread x 32 rows (x 2 panel slots when rows_per_thread
 * is 1 or 2) across all of n; its cost is the product's quad-padded blocks
 * per row.  The products' tiles are laid on one axis in list order; CTA b gets the
 * tiles whose first block falls in its contiguous range of that axis.  With
 * more than 8 products the host places the range boundaries so that the
 * largest range is as small as contiguous ranges allow (a binary search over
 * the bound, each step one greedy fill in list order); otherwise the axis is
 * split evenly.  No counterpart in the pages: it exposes the launcher's own
 * decision for inspection and testing.
 *   sms      : SMs to plan for (0 = the current device's count).
 *   plan     : HOST, receives rows per thread, grid, the total cost and the
 *              largest cost any CTA gets.
 *   cuts     : optional HOST int64 [max_cuts], receives the grid+1 range
 *              boundaries (as many as fit); may be NULL.
 * Returns Q1_OK or Q1_ERR_ARG. */
typedef struct q1_multi_plan {
  int rows_per_thread;    /* rows of a tile each consumer thread handles (1, 2 or 8) */
  int grid;               /* CTAs launched                                          */
  int64_t total_cost;     /* sum over products of tiles x padded blocks per row     */
  int64_t max_range_cost; /* largest tile cost owned by one CTA                     */
  int panel_warps;        /* 0: the streaming kernel above.  Else the call (up to
                             8 products of few rows in total) runs as one CTA per
                             panel_panels consecutive 32-row panels of a
                             product, whose panel_warps warps share out those
                             panels' blocks in units of panel_unit_blocks (grid
                             = ceil(panels / panel_panels) summed over the
                             products, rows_per_thread = 4, both costs 0, no
                             cuts) */
  int panel_unit_blocks;  /* 4 (quads) or 2 (half quads); 0 with the streaming kernel */
  int panel_panels;       /* panels a CTA takes: 1, or 2..8 when one CTA per panel
                             would put two or more panels on an SM (the CTA then
                             builds the activation table once for all of them);
                             0 with the streaming kernel */
} q1_multi_plan;

int q1_0_gemv_multi_plan(const q1_product *products, int count, int sms, q1_multi_plan *plan, int64_t *cuts,
                         int max_cuts);

/* Small-batch product ("kernels.rs -- the Q1_0 kernels", second bullet: each
 * lane's chain over the blocks is independent of every other chain, so one
 * stream of the weights serves several activation vectors, each vector's
 * chains kept apart): the matrix-vector product for each of nvec activation
 * vectors sharing one pass over the weights (1 <= nvec <= 64).
 *   q : device int8 [nvec][n]; d : device fp16 bits [nvec][n/32];
 *   out : device f32 [nvec][rows] (row-major per vector).
 * out[v][r] is bit-identical to q1_0_gemv on vector v. */
int q1_0_gemm_small(const void *packed, int64_t rows, int64_t n, int64_t nvec, const int8_t *q,
                    const uint16_t *d, float *out, void *stream);

/* Which kernel q1_0_gemm_small runs, for every call that follows in this
 * process (no counterpart in the pages: a tuning and testing knob).  Both
 * kernels give identical bits.
 *   choice : 0 = automatic (the default): from 8 vectors up, a cost model
 *            measured on a GB300 picks the faster of the two for the shape;
 *            1 = the dp4a kernel (CUDA cores) always;
 *            2 = the tensor-core kernel always (an f16 MMA gives each lane's
 *            sub-block chain in one exact f32 accumulator where an activation
 *            bound allows it, the dp4a chain elsewhere; it takes a per-call
 *            scratch of about 8 KB per 128 weights of n per 16 vectors from
 *            a pool the library keeps per device, and rejects shapes needing
 *            more than 64 MB).
 * Returns the previous choice, or Q1_ERR_ARG for another value. */
int q1_gemm_small_kernel(int choice);

/* Small-batch product that allocates no device memory.  The pages have no
 * counterpart: this is a service for callers, not part of the method.
 *
 * q1_0_gemm_small takes its tensor-core scratch from a memory pool at call
 * time.  Some callers cannot allow that: a serving loop that reserves all
 * device memory up front and forbids allocation on its decode path (an
 * allocation can stall behind other device work, and fails when a
 * framework's allocator already holds the memory), or a host whose memory
 * accounting must see every byte the process uses.  This call runs the
 * tensor-core kernel of q1_0_gemm_small with its scratch in one fixed array
 * of 8 MiB that the library holds in every device's memory from load to
 * process exit.  It calls no allocator.
 *   Arguments, layout and outputs: as q1_0_gemm_small (1 <= nvec <= 64);
 *   out[v][r] is bit-identical to q1_0_gemm_small's.
 *   Limit: the scratch needs 8 KB per 128 weights of n for each group of 16
 *   vectors, plus a few bytes; a larger n is rejected with Q1_ERR_ARG before
 *   anything is enqueued (for example n <= 32640 with 33..64 vectors,
 *   n <= 130944 with 1..16).
 *   First call on a device: it looks up the device address of the array on
 *   the current device (once per device); make that first call before any
 *   stream capture.
 *   Sharing: every call on a device uses the same array, and the array keeps
 *   the last call's contents (nothing in it needs to start at zero: each call
 *   writes what it reads).  Calls whose work overlaps on the GPU (on different
 *   streams, or from different host threads without ordering) race on it;
 *   order them, e.g. issue them on one stream.
 * Errors: Q1_ERR_ARG for a bad shape, pointer or a size beyond the limit;
 * Q1_ERR_CUDA for a failed lookup or launch. */
int q1_0_gemm_small_noalloc(const void *packed, int64_t rows, int64_t n, int64_t nvec, const int8_t *q,
                            const uint16_t *d, float *out, void *stream);

/* ---------------------------------------------------------------------------
 * Q2_0 (ternary) weights: the sibling format the pages name as the next GPU
 * kernel ("Advantages and efficiency", where optimization goes next;
 * "Limitations": no Q2_0 GPU kernel yet) without giving its layout or
 * arithmetic.  This library's reading:
 *   block (34 bytes) = fp16 scale d0 (little-endian), then 32 bytes of 2-bit
 *     codes: element j's code is (qs[j/4] >> 2*(j%4)) & 3, and codes 0, 1, 2
 *     mean the weights -d0, 0, +d0 (code 3 is not a weight);
 *   row product = the Q1_0 definition at the top of this file with the lane
 *     sum taken over ternary values: +1 contributes q, -1 the negation of q
 *     (-(-128) stays -128), 0 nothing.
 * Every output is bit-identical to that CPU definition.  Same conventions as
 * the Q1_0 calls.
 * ------------------------------------------------------------------------- */

/* Bytes of the packed Q2_0 buffer for a rows x n matrix (34 bytes per 128
 * weights, rows padded to a multiple of 256 and blocks per row to a multiple
 * of 4).  Host-only; negative Q1_ERR_ARG for a bad shape. */
int64_t q2_0_packed_bytes(int64_t rows, int64_t n);

/* Repack Q2_0 weights once into the library's device layout (two sign planes,
 * +1 and -1, in the Q1_0 bit order).
 *   blocks : device, rows*(n/128) consecutive 34-byte blocks, row-major, as
 *            above; only 2-byte alignment is required.
 *   packed : device, q2_0_packed_bytes(rows, n) bytes, written entirely.
 * Synchronous.  Returns Q1_ERR_ARG if any element holds the code 3 or any
 * block's fp16 scale is Inf or NaN (the message names the first such row and
 * block; the packed buffer must then not be used), or for a bad shape or
 * pointer.  Like q1_0_pack, the check uses device memory of this call alone. */
int q2_0_pack(const uint8_t *blocks, int64_t rows, int64_t n, void *packed, void *stream);

/* Inverse of q2_0_pack: writes rows*(n/128) 34-byte blocks identical to the
 * ones that were packed (codes 0..2). */
int q2_0_unpack(const void *packed, int64_t rows, int64_t n, uint8_t *blocks, void *stream);

/* Q2_0 matrix-vector product: as q1_0_gemv, with `packed` from q2_0_pack. */
int q2_0_gemv(const void *packed, int64_t rows, int64_t n, const int8_t *q, const uint16_t *d,
              float *out, void *stream);

/* Several independent Q2_0 products in one launch: as q1_0_gemv_multi, each
 * descriptor's `packed` from q2_0_pack(rows, n). */
int q2_0_gemv_multi(const q1_product *products, int count, void *stream);

/* q2_0_gemv_multi with the L2 prefetch of q1_0_gemv_multi_prefetch. */
int q2_0_gemv_multi_prefetch(const q1_product *products, int count, const q1_range *prefetch, int nranges,
                             void *stream);

/* The work split of a q2_0_gemv_multi launch: as q1_0_gemv_multi_plan.  The
 * kernel choice for a single product can differ from Q1_0's (the Q2_0 panel
 * kernel keeps more registers a thread, so fewer of its CTAs fit an SM). */
int q2_0_gemv_multi_plan(const q1_product *products, int count, int sms, q1_multi_plan *plan, int64_t *cuts,
                         int max_cuts);

/* Device status word of the library's kernels on the current device.  A
 * kernel whose bounded internal wait gives up (it never should: every wait is
 * for work the same kernel issued) sets bit 0 instead of hanging, and skips
 * its remaining output.  Synchronous: copies the word to the host.
 *   clear : nonzero resets the word to 0 after reading it.
 * Returns the status flags (0 = no event) or a negative Q1_ERR_CUDA. */
int q1_device_status(int clear);

/* On-card self-check ("How it is verified": verify_q1_0 compares every kernel
 * and shape with the CPU bits, including -128 quants and a layer-shaped regime
 * whose per-block scales make products inexact in f32; the Q2_0 product is
 * checked the same way).  Runs synchronously on
 * the current device with its own allocations, against a host-side reference
 * compiled into the library.
 *   flags  : 0 = default shape set (small products for the panel kernel, two
 *            with too many rows for it that take the streaming kernel, and
 *            the batched product through q1_0_gemm_small and, for its
 *            tensor-core kernel, q1_0_gemm_small_noalloc), preceded by an
 *            exhaustive check of the kernels' quantizer rounding (every
 *            float |t| < 2^22 against the device's roundf); bit 0 (1) =
 *            quick set (three small shapes, no
 *            rounding check);
 *            bit 1 (2) = negative control: in every one-vector case the
 *            packed scales of one row (nonzero reference output, about the
 *            middle row) are doubled after packing, so the check must report
 *            that row as the first differing one and return Q1_MISMATCH;
 *            bit 2 (4) = before the cases, run the library's bounded wait on an
 *            mbarrier nothing completes (20 ms limit): it must give up and let
 *            its kernel return, and the cases that follow show the device still
 *            works (the failure path of every product kernel's waits).
 *   report : host buffer receiving one line per kernel and shape, or the first
 *            differing row ("row i differs ..."); may be NULL.
 * Returns Q1_OK if every output is bit-identical, Q1_MISMATCH (2) if any
 * differs, or a negative error. */
int q1_0_verify(int flags, char *report, size_t report_len);

#ifdef __cplusplus
}
#endif

#endif /* Q1GEMV_H */
