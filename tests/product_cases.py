"""Copies whose source or destination is built by the products of
"CUTE布局代数" §4.1 (blocked_product, logical_product): (name, source,
destination, element bytes, the product-built side's closed form, the
planned paths).  Shared by the host and GPU tests."""

PRODUCT_CASES = [
    # a 64x64 bf16 tile (row-major) blocked over a 32x16 grid: the row-major
    # 2048x1024 matrix into tile-major order -- 64-element runs shared by
    # both sides (VEC)
    ("blocked_tile_grid_bf16", ("layout", (2048, 1024), (1024, 1)),
     ("blocked_product", ("layout", (64, 64), (64, 1)),
      ("layout", (32, 16), (16, 1))), 2,
     "((64,32),(64,16)):((64,65536),(1,4096))", ["VEC"]),
    # the same tiling from a column-major fp32 source: a transpose into the
    # tiles (STAGED)
    ("blocked_tile_grid_xpose_f32", ("layout", (2048, 1024), (1, 2048)),
     ("blocked_product", ("layout", (64, 64), (64, 1)),
      ("layout", (32, 16), (16, 1))), 4,
     "((64,32),(64,16)):((64,65536),(1,4096))", ["STAGED"]),
    # a destination with gaps: the logical product of a tile that uses 8 of
    # every 16 slots with a grid that uses 64 of every 128; slots outside
    # its image stay untouched (VEC over the 8-element runs)
    ("logical_product_gaps_f16", ("layout", (32, 16384), (1, 32)),
     ("logical_product", ("layout", (8, 4), (1, 16)),
      ("layout", (64, 256), (1, 128))), 2,
     "((8,4),((2,32),256)):((1,16),((8,64),4096))", ["VEC"]),
    # a source with gaps: a column-pitch-128 tile blocked over a gapped
    # grid, read into a row-major 1024x1024 destination (STAGED transpose)
    ("blocked_gapped_src_f32",
     ("blocked_product", ("layout", (64, 64), (1, 128)),
      ("layout", (16, 16), (1, 32))),
     ("layout", (1024, 1024), (1024, 1)), 4,
     "((64,(2,8)),(64,16)):((1,(64,8192)),(128,131072))", ["STAGED"]),
]
