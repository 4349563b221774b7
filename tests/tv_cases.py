"""Thread-value tile copy cases shared by the host replay and the GPU
parity tests: (name, src, smem, dst, thread layout of the load phase, of
the store phase, element bytes, expected plan choices)."""


def zd(shape, stride, tile):
    return ("zipped_divide", ("layout", shape, stride), tile)


CASES = [
    # name, src, smem, dst, thr_load, thr_store, eb, expected choices
    ("transpose_f32_plain",
     zd((256, 192), (1, 256), (32, 32)), ("layout", (32, 32), (1, 32)),
     zd((256, 192), (192, 1), (32, 32)), "(8,32):(1,8)", "(32,8):(8,1)", 4,
     {"load.vec_bytes": 16, "store.vec_bytes": 4}),
    ("transpose_f32_padded",
     zd((256, 192), (1, 256), (32, 32)), ("layout", (32, 32), (1, 33)),
     zd((256, 192), (192, 1), (32, 32)), "(32,8):(1,32)", "(8,32):(32,1)", 4,
     {"load.vec_bytes": 4, "store.smem_wavefronts": 32}),
    ("transpose_f32_swizzled",
     zd((256, 192), (1, 256), (32, 32)),
     ("swizzle", 3, 2, 5, ("layout", (32, 32), (1, 32))),
     zd((256, 192), (192, 1), (32, 32)), "(8,32):(1,8)", "(32,8):(8,1)", 4,
     {"load.vec_bytes": 16}),
    ("tiles_swizzled_bf16",
     zd((512, 384), (384, 1), (64, 64)),
     ("swizzle", 3, 3, 6, ("layout", (64, 64), (64, 1))),
     ("swizzle", 3, 4, 3,
      ("layout", ((64, 64), (8, 6)), ((64, 1), (24576, 4096)))),
     "(32,8):(8,1)", "(32,8):(8,1)", 2,
     {"load.vec_bytes": 16, "store.vec_bytes": 16,
      "load.smem_wavefronts": 64, "store.smem_wavefronts": 64}),
    ("nhwc_to_nchw_f16",   # tile (hw 56, c 64), grid (hw tiles 8, n 4)
     ("layout", ((56, 64), (8, 4)), ((64, 1), (3584, 28672))),
     ("layout", (56, 64), (64, 1)),
     ("layout", ((56, 64), (8, 4)), ((1, 448), (56, 28672))),
     "(8,8):(8,1)", "(56,4):(1,56)", 2,
     {"load.vec_bytes": 16, "load.values": 7, "store.vec_bytes": 2}),
    ("u8_ragged_grid",
     zd((96, 80), (1, 96), (32, 16)), ("layout", (32, 16), (16, 1)),
     zd((96, 80), (80, 1), (32, 16)), "(2,16):(16,1)", "(32,4):(1,32)", 1,
     None),
    ("b128_elements",
     zd((40, 24), (24, 1), (8, 8)), ("layout", (8, 8), (8, 1)),
     zd((40, 24), (1, 40), (8, 8)), "(8,8):(8,1)", "(8,8):(1,8)", 16,
     {"load.vec_bytes": 16}),
    ("f64_fewer_threads_store",
     zd((128, 64), (1, 128), (32, 32)), ("layout", (32, 32), (1, 32)),
     zd((128, 64), (64, 1), (32, 32)), "(16,16):(1,16)", "(32,2):(2,1)", 8,
     None),
    ("nested_tile_modes",  # tile modes (4,8) and 16, a grid of 12
     ("layout", (((4, 8), 16), 12), (((1, 4), 32), 512)),
     ("layout", ((4, 8), 16), ((1, 4), 32)),
     ("layout", (((4, 8), 16), 12), (((128, 1), 8), 512)),
     "(8,16):(1,8)", "((4,8),4):((1,4),32)", 4,
     {"load.vec_bytes": 16, "store.vec_bytes": 4}),
    # a destination swizzle reaching above the tile bases: applied to the
    # whole offset per value, not folded into the in-tile offsets
    ("tiles_wide_swizzle_bf16",
     zd((512, 384), (384, 1), (64, 64)),
     ("swizzle", 3, 3, 6, ("layout", (64, 64), (64, 1))),
     ("swizzle", 2, 3, 13,
      ("layout", ((64, 64), (8, 6)), ((64, 1), (24576, 4096)))),
     "(32,8):(8,1)", "(32,8):(8,1)", 2,
     {"load.vec_bytes": 16, "store.vec_bytes": 16}),
    # the layouts bench.py times on the 4096x4096 fp32 transpose, smaller
    ("bench_transpose_scalar_xor5",
     zd((320, 192), (1, 320), (64, 64)),
     ("swizzle", 5, 0, 6, ("layout", (64, 64), (1, 64))),
     zd((320, 192), (192, 1), (64, 64)), "(32,8):(1,32)", "(8,32):(32,1)", 4,
     {"load.vec_bytes": 4, "store.vec_bytes": 4,
      "load.smem_wavefronts": 128, "store.smem_wavefronts": 128}),
    ("bench_transpose_vector_loads",
     zd((320, 192), (1, 320), (64, 64)),
     ("swizzle", 3, 2, 6, ("layout", (64, 64), (1, 64))),
     zd((320, 192), (192, 1), (64, 64)), "(16,16):(1,16)", "(8,32):(32,1)", 4,
     {"load.vec_bytes": 16, "store.smem_wavefronts": 512}),
]
