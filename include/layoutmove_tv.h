/* layoutmove_tv.h -- arguments of the thread-value partitioned tile copy.
 *
 * A tile copy through shared memory in two phases, each a local_partition
 * of the tile by a thread layout ("CUTLASS Layout可视化" §5.3: a thread's
 * fragment of a shared tile is local_partition(sA, thread_layout,
 * thread_idx); "CUTE布局代数" §5.1: the global-to-shared copy is
 * make_copy(gmem_layout, smem_layout)).  The load phase moves the tile from
 * the source layout into the shared layout, the store phase from the shared
 * layout to the destination layout.  Each phase groups `vec` consecutive
 * coordinates of one tile mode into a vector, partitions the grouped tile by
 * its thread layout and gives thread t, for its value v, the byte offsets
 *     from = base_from(t) + from_val[v],   to = base_to(t) + to_val[v]
 * (before the side's swizzle), where base(t) sums, over the thread layout's
 * leaves j, ((t / leaf_stride[j]) % leaf_ext[j]) * step[j].  Every offset,
 * step and stride below is in bytes, and every swizzle acts on byte
 * offsets (an element swizzle Swizzle<B,M,S> becomes <B, M+log2(eb), S>).
 *
 * lm_tv_plan_args (layoutmove.h) fills this struct on the host; the device
 * functions of layoutmove_tv.cuh read it.  Plain C, no CUDA types: a
 * consumer kernel takes it as a `const __grid_constant__ lm_tv_args`
 * parameter (about 2.7 KB).
 */
#ifndef LAYOUTMOVE_TV_H
#define LAYOUTMOVE_TV_H

#include <stdint.h>

#define LM_TV_MAX_THR_LEAVES 6   /* thread-layout leaves of extent > 1   */
#define LM_TV_MAX_VALUES 128     /* vectors per thread per tile           */
#define LM_TV_MAX_GRID 8         /* joint modes of the grid of tiles      */

/* Division by an invariant divisor d (1 <= d < 2^31) with a multiply and
 * shifts (Granlund & Montgomery, "Division by invariant integers using
 * multiplication", PLDI 1994, round-up method): for any 32-bit n,
 * t = mulhi(m, n), n / d = (t + ((n - t) >> s1)) >> s2. */
typedef struct lm_tv_fastdiv {
  uint32_t d, m, s1, s2;
} lm_tv_fastdiv;

typedef struct lm_tv_phase {
  int32_t n_thr;       /* threads 0 .. n_thr-1 take part                 */
  int32_t n_val;       /* vectors each of them moves per tile            */
  int32_t vec_bytes;   /* bytes per vector: 1, 2, 4, 8 or 16             */
  int32_t n_leaves;    /* thread-layout leaves used by base(t)           */
  int32_t leaf_ext[LM_TV_MAX_THR_LEAVES];
  int32_t leaf_stride[LM_TV_MAX_THR_LEAVES];
  int32_t from_step[LM_TV_MAX_THR_LEAVES];  /* bytes per coordinate unit    */
  int32_t to_step[LM_TV_MAX_THR_LEAVES];
  int32_t from_val[LM_TV_MAX_VALUES];       /* bytes past base_from(t)      */
  int32_t to_val[LM_TV_MAX_VALUES];         /* bytes past base_to(t)        */
} lm_tv_phase;

typedef struct lm_tv_args {
  int32_t elem_bytes;     /* 1, 2, 4, 8 or 16                               */
  int32_t smem_bytes;     /* bytes of the shared tile (dynamic shared mem.) */
  int32_t block_threads;  /* max of the phases' n_thr, rounded up to 32     */
  int32_t n_grid;         /* joint modes of the grid of tiles               */
  int64_t n_tiles;
  int64_t grid_ext[LM_TV_MAX_GRID];  /* tile index: colex over these        */
  int64_t grid_src[LM_TV_MAX_GRID];  /* bytes per grid coordinate, src      */
  int64_t grid_dst[LM_TV_MAX_GRID];  /* bytes per grid coordinate, dst      */
  lm_tv_fastdiv grid_div[LM_TV_MAX_GRID];  /* by grid_ext, when grid_fast   */
  int32_t src_swz[3];     /* Swizzle<B,M,S> of each side on byte offsets;
                             B == 0: none                                   */
  int32_t smem_swz[3];
  int32_t dst_swz[3];
  int32_t grid_fast;      /* n_tiles < 2^32 and every grid_ext < 2^31: tile
                             coordinates by grid_div in 32 bits             */
  int32_t src_swz_tile;   /* 1: src_swz commutes with adding a tile base (no
                             swizzle, or every grid stride a multiple of
                             2^(B+M+S) bytes), so it may be applied to the
                             in-tile offset alone                           */
  int32_t dst_swz_tile;   /* the same for dst_swz                           */
  int32_t offsets32;      /* 1: every in-tile byte offset fits 31 bits      */
  lm_tv_phase load;       /* source (global) -> shared tile                 */
  lm_tv_phase store;      /* shared tile -> destination (global)            */
} lm_tv_args;

#endif /* LAYOUTMOVE_TV_H */
