/*
 * layoutmove.h -- C ABI of the GB300 layout-driven data movement library.
 *
 * A layout is a function from a logical coordinate to an element offset,
 * written shape:stride with nested modes, e.g. ((4,2),(2,4)):((2,16),(1,8)):
 * the offset is the inner product of the coordinate with the strides
 * ("CUTLASS Layout可视化：从print_layout理解GPU内存映射与性能优化" §2.1, §3.2;
 * "CUTE布局代数：GPU张量计算的内存优化革命" §2.1).  Optionally the affine
 * offset then passes through an XOR Swizzle<B,M,S> ("CUTLASS Layout可视化"
 * §4.3).  A copy moves a tensor from one layout to another over the same
 * logical coordinates: out[dst(i)] = in[src(i)] for every logical index i
 * ("CUTE布局代数" §5.1, make_copy(gmem_layout, smem_layout)).
 *
 * Conventions that hold for every function below:
 *  - Offsets, strides, sizes and capacities count ELEMENTS, not bytes
 *    (the PitchLinearStripminedThreadMap article, hotelren.com, §1.2).
 *  - A 1-D logical index is split over the leaves first-leaf-fastest
 *    ("colex"): the leaves of mode 0 before those of mode 1, the first leaf
 *    of each mode fastest.
 *  - Extents are >= 0, strides >= 0; an extent of 0 makes an empty layout
 *    (size 0, cosize 0) whose copy enqueues nothing.  All arithmetic is
 *    int64 and checked:
 *    a result that does not fit returns LM_E_OVERFLOW.
 *  - Every function returns an lm_status (LM_OK = 0, errors < 0) except the
 *    destroy functions and the string lookups.  No function aborts, exits or
 *    lets a C++ exception cross this boundary.  On error, output handles are
 *    set to NULL and output scalars are left unchanged.
 *  - Handles are immutable after creation; they may be shared between
 *    threads.  The caller owns every handle it receives and frees it with the
 *    matching destroy function (NULL is accepted and ignored).
 *  - Device buffers are owned by the caller and must stay valid until the
 *    stream has finished the work enqueued on them.
 */
#ifndef LAYOUTMOVE_H
#define LAYOUTMOVE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lm_layout lm_layout; /* opaque, freed by lm_layout_destroy */
typedef struct lm_plan lm_plan;     /* opaque, freed by lm_plan_destroy   */
typedef struct lm_tv_plan lm_tv_plan; /* opaque, freed by lm_tv_plan_destroy */
typedef struct lm_exchange lm_exchange; /* opaque, lm_exchange_destroy       */

typedef enum lm_status {
  LM_OK = 0,
  LM_E_INVALID = -1,           /* malformed argument (NULL, bad extent, ...)  */
  LM_E_INCOMPATIBLE = -2,      /* src and dst sizes differ                    */
  LM_E_NOT_REPRESENTABLE = -3, /* the algebraic result is no shape:stride
                                  (+swizzle) layout: divisibility fails, or
                                  the inner layout of a composition is
                                  swizzled                                    */
  LM_E_NOT_INJECTIVE = -4,     /* destination not shown to be one-to-one      */
  LM_E_OVERFLOW = -5,          /* int64 overflow in sizes or offsets          */
  LM_E_CAPACITY = -6,          /* a buffer is smaller than the layout needs   */
  LM_E_OVERLAP = -7,           /* src and dst byte ranges overlap             */
  LM_E_CUDA = -8,              /* a CUDA call failed; see lm_last_cuda_error  */
  LM_E_TIMEOUT = -9,           /* a bounded device wait gave up (see
                                  lm_device_status)                           */
  LM_E_NOMEM = -10,            /* host allocation failed                      */
  LM_E_BUFFER = -11            /* a text output buffer is too small           */
} lm_status;

/* ---------------------------------------------------------------------------
 * Layout construction and inspection (host only)
 * ------------------------------------------------------------------------- */

/* Build shape:stride from its leaves.  leaves_per_mode[m] leaves form
 * top-level mode m (n_modes modes, the counts summing to n_leaves); a mode of
 * one leaf is a plain integer mode, a mode of several leaves a nested tuple.
 * n_modes == 0 means one flat mode holding all leaves as an integer
 * (n_leaves must then be 1).  Example: ((4,2),(2,4)):((2,16),(1,8)) is
 * n_leaves=4, shape={4,2,2,4}, stride={2,16,1,8}, n_modes=2,
 * leaves_per_mode={2,2}.  ("CUTE布局代数" §2.1.)
 * Errors: LM_E_INVALID (NULL, extent < 1, stride < 0, counts that do not add
 * up), LM_E_OVERFLOW. */
int lm_layout_make(int n_leaves, const int64_t* shape, const int64_t* stride,
                   int n_modes, const int* leaves_per_mode, lm_layout** out);

/* Parse the printed notation, any nesting depth: "8:1", "(4,2):(2,1)",
 * "((4,2),(2,4)):((2,16),(1,8))", static marks accepted ("(4,2):(_2,_1)",
 * "CUTLASS Layout可视化" §3.2), and a swizzle prefix
 * "Sw<3,4,3> o ((64,64),(128,128)):((64,1),(524288,4096))".
 * Errors: LM_E_INVALID with no partial result. */
int lm_layout_parse(const char* text, lm_layout** out);

/* Print the same notation (no static marks).  Writes a NUL-terminated string
 * into buf; LM_E_BUFFER if cap is too small (buf then holds a truncated,
 * NUL-terminated prefix when cap > 0). */
int lm_layout_to_string(const lm_layout* layout, char* buf, size_t cap);

/* size = product of all extents.  cosize = one past the largest offset of
 * the affine part; with a swizzle, rounded up to a multiple of 2^(M+B), the
 * smallest bound that holds every swizzled offset whatever the layout.  A
 * buffer of cosize elements holds every offset. */
/* print_layout ("CUTLASS Layout可视化" §3.1, §4.1): a rank-2 layout as a
 * grid, one line per mode-0 coordinate (row), one column per mode-1
 * coordinate, each entry the offset (swizzle applied) right-aligned to a
 * common width.  With bank_elem_bytes > 0 each entry is instead the shared-
 * memory bank of the element, (offset * bank_elem_bytes / 4) mod 32: the
 * "take every offset mod 32" check of §6.4, printed.  Buffer rules as
 * lm_layout_to_string.  Errors: LM_E_INVALID (NULL, rank != 2, more than
 * 2^16 entries, bank_elem_bytes outside 0..16), LM_E_BUFFER. */
int lm_layout_print_grid(const lm_layout* layout, int bank_elem_bytes,
                         char* buf, size_t cap);

int lm_layout_size(const lm_layout* layout, int64_t* size);
int lm_layout_cosize(const lm_layout* layout, int64_t* cosize);

/* Number of top-level modes and of leaves; the leaves themselves (shape and
 * stride arrays of at least n_leaves entries, either may be NULL); the
 * swizzle (b = 0 when there is none).  leaves_per_mode may be NULL. */
int lm_layout_rank(const lm_layout* layout, int* n_modes, int* n_leaves);
int lm_layout_leaves(const lm_layout* layout, int64_t* shape, int64_t* stride,
                     int* leaves_per_mode);
int lm_layout_get_swizzle(const lm_layout* layout, int* b, int* m, int* s);

/* offset = L(i) for a colex index 0 <= i < size, swizzle included.
 * Errors: LM_E_INVALID for i out of range. */
int lm_layout_eval(const lm_layout* layout, int64_t index, int64_t* offset);

/* offset = swizzle(sum_k coord[k] * stride[k]) for a full leaf coordinate
 * (n == number of leaves).  No bounds check on the coordinates: this is the
 * bare offset formula of "CUTLASS Layout可视化" §2.1, under which the
 * blocked layout's printed sample of "CUTE布局代数" §6.1 reads
 * (r, c) -> 2r + 16c as leaf coordinate (r, c, 0, 0).
 * Errors: LM_E_INVALID (n mismatch, negative coordinate), LM_E_OVERFLOW. */
int lm_layout_eval_coord(const lm_layout* layout, int n,
                         const int64_t* leaf_coord, int64_t* offset);

/* ---------------------------------------------------------------------------
 * Layout algebra (host only)
 * ------------------------------------------------------------------------- */

/* R = A o B, R(i) = A(B(i)), shaped like B ("CUTE布局代数" §2.2, §3.1).  B's
 * value is read by A as a colex index; past A's last extent A's last leaf
 * keeps counting.  A may carry a swizzle (it stays outermost in R).
 * Example: (8,8):(1,9) o ((4,8),2):((16,1),8) = ((4,8),2):((18,1),9).
 * Errors: LM_E_NOT_REPRESENTABLE when B is swizzled or a B stride/extent does
 * not divide A's leaf structure; LM_E_OVERFLOW. */
int lm_layout_compose(const lm_layout* a, const lm_layout* b, lm_layout** r);

/* zipped_divide(L, tiler) ("CUTE布局代数" §3.2): n must equal L's number of
 * top-level modes; tiler[k] consecutive coordinates of mode k form a tile.
 * Result ((tile_0,...,tile_n-1),(rest_0,...,rest_n-1)), each piece the mode
 * composed with t:1 (tile) and (n_k/t_k):t_k (rest); L's swizzle is kept.
 * Example: (128,128):(1,128) / (4,8) = ((4,8),(32,16)):((1,128),(4,1024)).
 * Errors: LM_E_INVALID (n mismatch, tiler < 1), LM_E_NOT_REPRESENTABLE
 * (a tiler entry that does not divide its mode, or a mode whose leaves it
 * cannot split). */
int lm_layout_zipped_divide(const lm_layout* layout, int n,
                            const int64_t* tiler, lm_layout** r);

/* R = Swizzle<B,M,S> o L: offsets o -> o ^ ((o >> S) & ((2^B - 1) << M))
 * ("CUTLASS Layout可视化" §4.3; Swizzle<3,0,3> on (8,8):(8,1) is the page's
 * row*8 + (col ^ row)).  Requires B >= 0, M >= 0, S >= B, B+M+S <= 40.
 * Errors: LM_E_INVALID, LM_E_NOT_REPRESENTABLE (L already swizzled). */
int lm_layout_swizzle(const lm_layout* layout, int b, int m, int s,
                      lm_layout** r);

/* R = (A, B): A's modes become mode 0, B's mode 1, so B is the slower
 * (batch) mode.  Errors: LM_E_NOT_REPRESENTABLE if either is swizzled. */
int lm_layout_concat(const lm_layout* a, const lm_layout* b, lm_layout** r);

/* Flat layout with the same function: extent-1 leaves dropped, neighbours
 * (e0:d0, e1:d1) with d1 == e0*d0 merged.  Swizzle kept. */
int lm_layout_coalesce(const lm_layout* layout, lm_layout** r);

/* Right inverse L‡ ("CUTE布局代数" §2.3): the layout R with L(R(j)) = j for
 * 0 <= j < size(R), where size(R) is the length of the contiguous run of
 * offsets 0, 1, 2, ... that L reaches (size(L) for a bijection onto
 * [0, size)).  Errors: LM_E_NOT_REPRESENTABLE for a swizzled L. */
int lm_layout_right_inverse(const lm_layout* layout, lm_layout** r);

/* K = max{k : A‡(j) = B‡(j) for all j < k} ("CUTE布局代数" §2.3): the number
 * of leading offsets at which both layouts hold the same logical element.
 * Offsets with no or several preimages end the run.
 * Errors: LM_E_INCOMPATIBLE (sizes differ). */
int lm_layout_max_common_vector(const lm_layout* a, const lm_layout* b,
                                int64_t* k);

/* complement(L, cotarget): the layout R, strides increasing, with (L, R)
 * one-to-one and reaching every offset below cotarget when L's strides nest.
 * Walking L's leaves by increasing stride d (extent e), the gap between the
 * offsets reached so far (c, starting at 1) and d becomes a leaf d/c : c,
 * then c = e*d; a last leaf ceil(cotarget/c) : c runs R up to cotarget.
 * The operation the products of "CUTE布局代数" §4.1 rest on.
 * Errors: LM_E_INVALID (cotarget < 1), LM_E_NOT_REPRESENTABLE (swizzled L,
 * a stride that does not nest: d not a multiple of c, or d < c). */
int lm_layout_complement(const lm_layout* layout, int64_t cotarget,
                         lm_layout** r);

/* logical_product(A, B) = (A, complement(A, size(A)*cosize(B)) o B): B
 * repeats A, its coordinates stepping over whole copies of A
 * ("CUTE布局代数" §4.1).  blocked_product(A, B): the same modes zipped, mode
 * k = (A's mode k, the product's mode k), so a rank-r tile A laid out in the
 * order of a rank-r grid B; the page's 4x8 tile over a 2x5 grid gives shape
 * ((4,2),(8,5)).  Errors: LM_E_INVALID (blocked: ranks differ),
 * LM_E_NOT_REPRESENTABLE (swizzled operands, complement or composition not
 * representable). */
int lm_layout_logical_product(const lm_layout* a, const lm_layout* b,
                              lm_layout** r);
int lm_layout_blocked_product(const lm_layout* a, const lm_layout* b,
                              lm_layout** r);

/* local_partition(layout, thr, thr_idx): the part of a tile that thread
 * thr_idx owns under the thread layout thr, as in the
 * local_partition(sA, thread_layout, thread_idx) call of "CUTLASS Layout
 * 可视化" §5.3.  thr must map its domain one-to-one onto [0, size(thr))
 * (strides 1, e0, e0*e1, ... in some order) and have rank <= rank(layout);
 * with T_k the size of thr's mode k (1 past its rank) and c the coordinate
 * thr maps to thr_idx, the thread owns the mode coordinates c_k + T_k*r_k.
 * *part is the layout of r (colex, no swizzle; the rest mode of
 * zipped_divide(layout, T)), *base the offset at r = 0, so value v sits at
 * Swz(*base + part(v)), Swz being layout's swizzle (none: identity).
 * Errors: LM_E_INVALID (NULL, thr not a compact bijection or swizzled,
 * thr_idx outside [0, size(thr)), rank(thr) > rank(layout)),
 * LM_E_NOT_REPRESENTABLE (a T_k does not divide mode k). */
int lm_layout_local_partition(const lm_layout* layout, const lm_layout* thr,
                              int64_t thr_idx, lm_layout** part,
                              int64_t* base);

/* The stripmined thread map of the PitchLinearStripminedThreadMap article
 * (hotelren.com, §2.2) as a layout over thread ids:
 * (pitch, strips, ceil(threads/(pitch*strips))):(1, k_row,
 * pitch*strips*k_row), whose colex evaluation is get_offset(thread_id).
 * Errors: LM_E_INVALID for arguments < 1. */
int lm_layout_stripmined(int64_t threads, int64_t pitch, int64_t strips,
                         int64_t k_row, lm_layout** r);

/* Shared-memory bank wavefronts of a warp-by-warp access pattern: the
 * check "CUTLASS Layout可视化" §5.2 and §6.4 ask of a tile layout (do one
 * warp's offsets, taken mod 32 banks, spread out?), counted.  Access i,
 * colex over the domain of `access`, is made by lane i % 32 of warp access
 * i / 32 and reads access_bytes at byte address access(i) * elem_bytes.
 * Model: 32 banks of 4 bytes; 16-byte accesses are served 8 lanes at a
 * time, 8-byte ones 16 at a time, narrower ones a whole warp at a time;
 * within such a group the cost is the largest number of distinct 4-byte
 * words that one bank holds (lanes reading one word share it).  *wavefronts
 * = the sum over all groups; *ideal = the conflict-free minimum, a group's
 * bytes over 128 (at least 1).  The copy planner chooses its shared tile's
 * pad and swizzle with the same model.
 * Errors: LM_E_INVALID (null pointers, elem_bytes or access_bytes not a
 * power of two in 1..16, size(access) > 2^24, an address not a multiple of
 * access_bytes or negative), LM_E_OVERFLOW. */
int lm_smem_wavefronts(const lm_layout* access, int elem_bytes,
                       int access_bytes, int64_t* wavefronts, int64_t* ideal);

/* Choose Pitch and Strips of the stripmined thread map (the
 * PitchLinearStripminedThreadMap article, hotelren.com, §2.2) for `threads`
 * threads, each moving vec_elems consecutive elements, over a tile of
 * `rows` rows of k_row elements of elem_bytes: the tile's rows lie ld
 * elements apart in global memory, and go to shared memory at smem(row,
 * col) (a rank-2 layout of sizes (rows, k_row), swizzle allowed; NULL:
 * row-major, k_row per row).  Thread t of the pass, with the map counted in
 * vectors (R = k_row / vec_elems per row), takes row (t/P)%S + (t/(P*S))*P*S
 * and vector column t%P.  Candidates: P and S powers of two, P <= R,
 * S <= rows, P*S <= threads, every thread's row inside the tile.  The
 * article's guidance (§4.1-§4.2: Pitch from the vector width and coalescing,
 * Strips against bank conflicts) becomes a cost, compared in this order:
 * the 128-byte global segments each warp touches (summed over warps,
 * *segments), the shared-memory wavefronts of the same accesses under the
 * bank model of lm_smem_wavefronts (*wavefronts), then the larger P, then
 * the larger S.  Errors: LM_E_INVALID (arguments out of range: threads not
 * in 1..1024, vec_elems not dividing k_row, vector bytes not a power of two
 * up to 16, ld < k_row, smem of other sizes, a misaligned shared address),
 * LM_E_NOT_REPRESENTABLE (no candidate keeps every thread inside the
 * tile). */
int lm_stripmined_tune(int64_t threads, int64_t k_row, int64_t rows,
                       int64_t ld, int elem_bytes, int vec_elems,
                       const lm_layout* smem, int64_t* pitch, int64_t* strips,
                       int64_t* segments, int64_t* wavefronts);

void lm_layout_destroy(lm_layout* layout);

/* ---------------------------------------------------------------------------
 * Copy plans and device work
 * ------------------------------------------------------------------------- */

/* Lower a src/dst layout pair into a copy plan for elements of elem_bytes in
 * {1, 2, 4, 8, 16}.  The plan refines both leaf lists to common modes,
 * coalesces and reorders them, checks that dst is injective, finds the
 * common contiguous run (the common vector of "CUTE布局代数" §2.3) and
 * chooses per piece of the domain a kernel: VEC (16-byte vectors along a run
 * both sides share), ZIP (a short interleave in registers), STAGED (tiles
 * staged through swizzled shared memory, loads contiguous along src, stores
 * contiguous along dst) or GENERIC (one element per thread).  The common
 * refinement is tried on each side's leaves as given and coalesced.  Pairs
 * without one are planned over each side's own leaves: GTILE (tiles through
 * shared memory, read along the source's unit-stride direction and written
 * along the destination's) when one side has unit stride along the logical
 * index and the other a unit-stride leaf behind at least 32 indices, else
 * GENERIC.  The plan is host data only; it holds no device memory and may
 * be used on any device and stream.
 * Errors: LM_E_INVALID, LM_E_INCOMPATIBLE (sizes differ),
 * LM_E_NOT_INJECTIVE (dst offsets could collide; proven exactly for every
 * layout up to 2^28 elements, otherwise by a sufficient test),
 * LM_E_OVERFLOW, LM_E_NOMEM. */
int lm_plan_copy(const lm_layout* src, const lm_layout* dst, int elem_bytes,
                 lm_plan** out);

/* Shard `rank` (0 <= rank < world) of the same copy, for running one copy on
 * several devices or streams: every logical index is independent, so the
 * shards need no exchange.  A pair with a common refinement is split along
 * its joint mode with the largest destination stride into `world` balanced
 * contiguous ranges (each shard writes one region of the destination; the
 * mode is the largest-stride one with at least `world` coordinates); other
 * pairs split the logical index range.  The shards of ranks 0..world-1
 * partition the copy exactly; each is an ordinary plan over the full
 * layouts (same buffers, same capacities).  world == 1 is lm_plan_copy.
 * Errors: as lm_plan_copy, and LM_E_INVALID for a bad rank or world. */
int lm_plan_copy_shard(const lm_layout* src, const lm_layout* dst,
                       int elem_bytes, int rank, int world, lm_plan** out);

/* One-line JSON description: pieces, path, modes, vector width, tile; the
 * element ranges of src and dst the copy can reach ("src_range",
 * "dst_range": [0, cosize) for a whole copy, the shard's own for a shard)
 * and whether no other shard writes inside the destination range
 * ("dst_own").  A GTILE piece also gives its parts' leaves as [extent,
 * byte stride] ("lo_leaves", "hi_leaves", "in_leaves") and the steps its
 * threads take between elements ("steps": per step its digits in the
 * part's mixed radix, "dstep" the byte offset change without carries and
 * "cadj" the extra change of a carry out of each leaf). */
int lm_plan_describe(const lm_plan* plan, char* buf, size_t cap);

/* Elements of src and dst that the plan reads and writes (sizes of their
 * layouts' domains are equal; this is that size), and the cosizes a buffer
 * must cover. */
int lm_plan_extent(const lm_plan* plan, int64_t* size, int64_t* src_cosize,
                   int64_t* dst_cosize);

/* Enqueue out[dst(i)] = in[src(i)] on cuda_stream (a cudaStream_t; NULL is
 * the legacy default stream).  src_dev/dst_dev are device pointers to
 * buffers of src_capacity_elems / dst_capacity_elems elements.  Host checks
 * before launch: capacities >= the layouts' cosizes (LM_E_CAPACITY), the byte
 * ranges [ptr, ptr + cosize*elem_bytes) do not overlap (LM_E_OVERLAP).  Base
 * pointers need only elem_bytes alignment: where a vector path needs 16-byte
 * alignment and the pointers lack it, the same plan runs with narrower
 * accesses.  Destination slots outside dst's image are not written.  The
 * call returns after enqueueing; it synchronises nothing.  A launch failure
 * returns LM_E_CUDA (lm_last_cuda_error has the cudaError_t).  For plans
 * whose description shows a STAGED piece with "bulk" set, LM_OK is
 * provisional: those kernels bound their waits on the device, and a wait
 * that gives up is reported only by lm_device_status, which a caller that
 * needs the result must check after the stream has reached the copy. */
int lm_layout_copy(const lm_plan* plan, const void* src_dev,
                   int64_t src_capacity_elems, void* dst_dev,
                   int64_t dst_capacity_elems, void* cuda_stream);

/* The same copy for buffers in host memory, through caller-provided device
 * staging buffers (src_dev / dst_dev, of src_capacity_elems /
 * dst_capacity_elems elements): enqueues on cuda_stream the upload of the
 * whole host source (src_capacity_elems elements), the copy of
 * lm_layout_copy between the staging buffers, and the download of the
 * destination's [0, cosize) into dst_host.  When the destination layout
 * does not cover every slot below its cosize, the host destination is
 * uploaded first, so slots outside the image come back unchanged.  A shard
 * (lm_plan_copy_shard) moves only the ranges its pieces reach
 * ("src_range" / "dst_range" of its description), so the shards of one
 * copy may run on separate streams over the same host and staging buffers
 * -- provided each owns its destination range ("dst_own"); a shard that
 * does not is refused with LM_E_INVALID.  Host buffers should be
 * page-locked for the transfers to be asynchronous.  Allocates nothing.
 * Errors: as lm_layout_copy (the staging buffers are the device buffers it
 * checks), LM_E_INVALID, LM_E_CUDA for a failed transfer. */
int lm_layout_copy_host(const lm_plan* plan, const void* src_host,
                        int64_t src_capacity_elems, void* dst_host,
                        int64_t dst_capacity_elems, void* src_dev,
                        void* dst_dev, void* cuda_stream);

/* Bytes of the fixed device staging area of lm_layout_copy_host_static
 * (32 MiB). */
#define LM_HOST_COPY_STATIC_BYTES (32u * 1024u * 1024u)

/* lm_layout_copy_host for callers that cannot allocate device memory: the
 * same upload, copy and download, staged through a fixed area inside the
 * library instead of caller-provided device buffers.  The source pages have
 * no counterpart; this is a convenience of the ABI.  It is for code that
 * has no way to obtain device memory: a library embedded in a program whose
 * memory manager owns the device's memory, or a path that cannot afford
 * cudaMalloc/cudaFree (cudaFree waits for the whole device).  The call
 * allocates nothing.
 *
 * The area is a __device__ array of LM_HOST_COPY_STATIC_BYTES that every
 * GPU which loads the library holds until the process exits.  The source
 * is staged at its start, the destination at the next 256-byte boundary
 * after src_capacity_elems * elem_bytes; a copy whose two parts do not fit
 * is refused with LM_E_CAPACITY before anything is enqueued.  The first
 * call on a device, with that device current, looks up the area's device
 * address (cudaGetSymbolAddress) and keeps it for later calls on that
 * device; make that first call before any stream capture.  The address
 * belongs to the device's context: after cudaDeviceReset this process must
 * not call the function again.  Every call on a device shares the one area, which keeps the
 * last call's bytes: calls whose work overlaps on the GPU (other streams,
 * other host threads) race and must be ordered by the caller.  No part of
 * the area needs to start cleared: every destination byte that comes back
 * is written by the copy or, when the destination layout leaves slots of
 * [0, cosize) uncovered, uploaded from dst_host first.  Arguments, host
 * buffer rules, shard rules and other errors are those of
 * lm_layout_copy_host. */
int lm_layout_copy_host_static(const lm_plan* plan, const void* src_host,
                               int64_t src_capacity_elems, void* dst_host,
                               int64_t dst_capacity_elems, void* cuda_stream);

/* Number of kernel launches lm_layout_copy makes for this plan. */
int lm_plan_launches(const lm_plan* plan, int* launches);

/* Enqueue table[i] = L(i) for 0 <= i < size(L) into a device table of
 * offset_bytes (4 or 8) entries; capacity counts entries and must be
 * >= size(L).  With offset_bytes == 4 every offset must fit in int32
 * (LM_E_OVERFLOW otherwise).  ("CUTLASS Layout可视化" §2.3: the offset of
 * every logical coordinate, in logical order.)  Returns LM_E_CUDA on launch
 * failure. */
int lm_layout_eval_device(const lm_layout* layout, void* table_dev,
                          int offset_bytes, int64_t capacity,
                          void* cuda_stream);

void lm_plan_destroy(lm_plan* plan);

/* ---------------------------------------------------------------------------
 * Relayouts whose source and destination are both sharded across ranks
 * ------------------------------------------------------------------------- */

/* Plan rank `rank` of `world` of out[dst(i)] = in[src(i)] when every rank
 * holds only part of the source and must produce only part of the
 * destination: with the joint modes of the pair (as lm_plan_copy forms
 * them), rank r holds the source elements of range r of the joint mode with
 * the largest source stride ("in" mode) and produces the destination
 * elements of range r of the mode with the largest destination stride
 * ("out" mode); ranges are balanced (coordinates e*r/world up to
 * e*(r+1)/world), and both modes need at least `world` coordinates: when
 * the largest-stride mode of either side is shorter, the call fails with
 * LM_E_INVALID rather than shard a faster mode (whose ranges would overlap
 * in memory).  The
 * local shard buffers hold the global layouts' offsets from the shard's
 * first to its last, rebased to 0 (src_local / dst_local elements; for the
 * row-sharded transpose of a row-major matrix, the rows themselves).  Rank
 * p sends rank q the box where p's input range meets q's output range,
 * packed contiguously in the joint modes' colex order; the exchange is one
 * all-to-all of those buffers, done by the caller's collective.  The pages
 * do not shard: this is the copy of "CUTE布局代数" §5.1 (make_copy of a
 * layout pair) split over ranks, and only the placement of the shards
 * needs the exchange, every logical index being independent.
 * Errors: LM_E_INVALID (NULL, elem_bytes, rank/world, an empty copy, a
 * largest-stride mode with fewer than `world` coordinates on either side),
 * LM_E_INCOMPATIBLE (sizes differ or
 * no common refinement), LM_E_NOT_REPRESENTABLE (a swizzled side),
 * LM_E_NOT_INJECTIVE. */
int lm_plan_exchange(const lm_layout* src, const lm_layout* dst,
                     int elem_bytes, int rank, int world, lm_exchange** out);

/* JSON: joint modes, in/out modes, the local shard extents, and per peer
 * the box sent and received (count, base offset, modes). */
int lm_exchange_describe(const lm_exchange* x, char* buf, size_t cap);

/* Elements of the local source and destination shards, and per peer
 * (arrays of `world`, either may be NULL) the elements sent and received. */
int lm_exchange_sizes(const lm_exchange* x, int64_t* src_local,
                      int64_t* dst_local, int64_t* send_counts,
                      int64_t* recv_counts);

/* Enqueue the pack of the box bound for `peer` from the local source shard
 * into `send` (its compact image), or the unpack of the box received from
 * `peer` into the local destination shard: layout copies through
 * lm_layout_copy, with its buffer rules.  A peer with nothing to exchange
 * is a no-op.  Errors: LM_E_INVALID, LM_E_CAPACITY, LM_E_OVERLAP,
 * LM_E_CUDA. */
int lm_exchange_pack(const lm_exchange* x, int peer, const void* src_local,
                     int64_t src_capacity_elems, void* send,
                     int64_t send_capacity_elems, void* cuda_stream);
int lm_exchange_unpack(const lm_exchange* x, int peer, const void* recv,
                       int64_t recv_capacity_elems, void* dst_local,
                       int64_t dst_capacity_elems, void* cuda_stream);

/* All of this rank's packs, into one buffer holding the boxes for peers
 * 0..world-1 one after another (each box compact, as lm_exchange_pack
 * writes it; the send counts give the offsets), and all of its unpacks from
 * one buffer laid out the same way by sender.  When both the in and the out
 * mode split evenly over the ranks (every box the same shape) and differ,
 * each is a single layout copy ("one_copy_per_side" in the description);
 * otherwise one copy per peer.  Errors: as lm_exchange_pack/unpack. */
int lm_exchange_pack_all(const lm_exchange* x, const void* src_local,
                         int64_t src_capacity_elems, void* send,
                         int64_t send_capacity_elems, void* cuda_stream);
int lm_exchange_unpack_all(const lm_exchange* x, const void* recv,
                           int64_t recv_capacity_elems, void* dst_local,
                           int64_t dst_capacity_elems, void* cuda_stream);

void lm_exchange_destroy(lm_exchange* x);

/* ---------------------------------------------------------------------------
 * Thread-value partitioned tile copies through shared memory
 * ------------------------------------------------------------------------- */

/* Plan a copy out[dst(i)] = in[src(i)] that stages every tile in shared
 * memory with caller-chosen layouts: the global-to-shared copy
 * make_copy(gmem_layout, smem_layout) of "CUTE布局代数" §5.1, each thread
 * moving its local_partition of the tile ("CUTLASS Layout可视化" §5.3).
 * src and dst: layouts over the same domain whose mode 0 is the tile (its
 * own modes are the tile modes, as zipped_divide returns) and whose other
 * top modes number the tiles; the grid modes are refined jointly.  smem:
 * the shared tile, one mode per tile mode with the same sizes, injective,
 * at most 232448 bytes, swizzle allowed.  thr_load / thr_store: thread
 * layouts (compact bijections onto [0, size), at most 1024 threads, rank
 * at most the tile's) of the load phase (src -> smem) and the store phase
 * (smem -> dst).  A phase moves vectors of vec_*_bytes (0: the widest of
 * 16, 8, ..., elem_bytes that works) along one tile mode: that many
 * consecutive coordinates must be contiguous and aligned on both of its
 * sides; the thread layout then partitions the tile with that mode counted
 * in vectors, at most 128 vectors per thread.  A NULL thread layout asks
 * for the tuned one: the stripmined map of the PitchLinearStripminedThreadMap
 * article (§2.2) with Pitch and Strips chosen as lm_stripmined_tune chooses
 * them (§4.1-§4.2: fewest 128-byte global segments per warp, then fewest
 * shared-memory wavefronts), where the phase's global side gives the row
 * (its unit-stride tile mode, else mode 0; the other mode counts rows) and
 * the search keeps to maps whose one Pitch x Strips group holds every
 * thread with Pitch and Strips dividing the tile, the ones a thread layout
 * can express: (Pitch, Strips):(1, Pitch) along (row, rows), up to 256
 * threads, on tiles of rank 1 or 2.  lm_tv_plan_describe gives the
 * choices (the thread layouts, and Pitch, Strips and segments when tuned)
 * and the shared-memory wavefronts the bank model of lm_smem_wavefronts
 * predicts per tile for each phase.
 * Errors: LM_E_INVALID (NULL src/smem/dst/out, elem_bytes, limits above,
 * empty tile, a NULL thread layout for a tile of rank above 2),
 * LM_E_INCOMPATIBLE (sizes or tile modes differ, grids do not refine),
 * LM_E_NOT_INJECTIVE (smem or dst), LM_E_NOT_REPRESENTABLE (no vector
 * width fits, a thread extent does not divide its mode, or the offsets are
 * not base(thread) + value-offset), LM_E_OVERFLOW. */
int lm_tv_plan_create(const lm_layout* src, const lm_layout* smem,
                      const lm_layout* dst, const lm_layout* thr_load,
                      const lm_layout* thr_store, int elem_bytes,
                      int vec_load_bytes, int vec_store_bytes,
                      lm_tv_plan** out);

/* JSON description of a plan (same buffer rules as lm_plan_describe). */
int lm_tv_plan_describe(const lm_tv_plan* plan, char* buf, size_t cap);

/* Copy the plan's lm_tv_args (layoutmove_tv.h) into args, cap bytes long,
 * for consumer kernels that call the device functions of layoutmove_tv.cuh.
 * Errors: LM_E_INVALID, LM_E_BUFFER (cap < sizeof(lm_tv_args)). */
int lm_tv_plan_args(const lm_tv_plan* plan, void* args, size_t cap);

/* Enqueue the copy on cuda_stream: one block per tile at a time, the load
 * phase, a barrier, the store phase.  Buffers as for lm_layout_copy; src
 * must be aligned to the load phase's vector bytes and dst to the store
 * phase's.  Errors: LM_E_INVALID, LM_E_CAPACITY, LM_E_OVERLAP, LM_E_CUDA. */
int lm_tv_copy(const lm_tv_plan* plan, const void* src_dev,
               int64_t src_capacity_elems, void* dst_dev,
               int64_t dst_capacity_elems, void* cuda_stream);

void lm_tv_plan_destroy(lm_tv_plan* plan);

/* Static, NUL-terminated name of a status code. */
const char* lm_status_string(int status);

/* The cudaError_t of the last LM_E_CUDA returned on this thread (0 if
 * none). */
int lm_last_cuda_error(void);

/* Synchronise cuda_stream (a cudaStream_t, NULL for the legacy stream),
 * then report in *status whether a kernel of this library on the current
 * device gave up a bounded wait since the last reset: LM_OK, or
 * LM_E_TIMEOUT (the bulk-copy STAGED kernels bound every mbarrier wait at
 * about a second; a block that gives up records it here, waits -- again
 * bounded, about four seconds per stage -- for its own copies still in
 * flight, and exits, leaving its part of the destination unwritten).  If
 * even that drain runs out (copies from global memory that do not complete
 * in seconds mean the memory system has failed), the block has exited with
 * bulk copies still writing into shared memory it no longer owns, which can
 * corrupt a later block on that SM: after LM_E_TIMEOUT treat every result
 * on the device since the last reset as suspect.  The record is per device,
 * shared by every stream and sticky; reset != 0 clears it after reading.
 * Errors: LM_E_INVALID (NULL status), LM_E_CUDA. */
int lm_device_status(void* cuda_stream, int reset, int* status);

/* Self-test of the bounded device wait (no counterpart on the source
 * pages).  Clears the status record, launches one warp that waits on an
 * mbarrier -- with arrive == 0 nothing ever arrives, so the wait gives up
 * after about a second -- and returns the resulting status in *status
 * (LM_E_TIMEOUT when arrive == 0, LM_OK otherwise), clearing the record
 * again.  Never hangs and never faults; blocks the calling thread for about
 * a second when arrive == 0.  Errors: LM_E_INVALID, LM_E_CUDA. */
int lm_selftest_bounded_wait(int arrive, void* cuda_stream, int* status);

/* Library version, "major.minor.patch". */
const char* lm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LAYOUTMOVE_H */
