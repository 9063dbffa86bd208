"""Shapes of the GPU parity tests, shared with the CPU test that checks that every
kernel variant the planner can choose is exercised by at least one of them."""

EDGE = [
    ((2, 3), 1),
    ((1, 1, 1), 1),
    ((37, 41), 257),
    ((5, 7, 9, 11), 13),
    ((3,) * 8, 5),
    ((130, 3, 65), 130),
    ((1000, 2), 3),
    ((2, 1000), 4),
    ((64, 64, 64), 4),
    ((20, 20, 20, 20), 128),
    ((33, 17, 129), 64),
    ((128, 1, 128), 32),
    ((8, 200, 6), 200),
    ((129, 129, 7), 129),
    # shapes the tensor-core path takes: row and column tails, inner groups with
    # a p-side part, contraction lengths that are not multiples of 16 or 128
    ((200, 48, 40), 300),
    ((256, 12, 16, 8), 96),
    ((128, 128, 64), 17),
    ((96, 40, 36), 1000),
    ((160, 4, 4, 4, 4), 48),
    # small I_k: several pre indices stacked in one 128-row tensor-core tile
    ((24, 30, 40, 16), 96),
    ((16, 64, 40), 200),
    ((60, 8, 8, 36), 64),
    ((17, 33, 48), 130),
    # small I_k in the innermost mode (I_k * 4 bytes a multiple of 16): the
    # staging box holds several pre indices and is transposed into one tile
    ((30, 40, 20), 96),
    ((12, 50, 36), 64),
    ((7, 9, 11, 44), 130),
    ((5, 6, 40, 28), 260),
    # large R: the A operand staged in tensor memory (224-column tiles), K-major
    # and innermost modes, row / column / contraction tails
    ((24, 40, 136), 460),
    ((130, 6, 7, 100), 500),
    # K-major modes on the fp16-image kernel (Y split once into fp16 images):
    # a contraction tail inside the last 64-index step, row and column tails,
    # 128- and 256-column tiles, pre modes on one or both sides of the mode
    ((136, 24, 120), 260),
    ((200, 96, 64), 300),
    ((160, 8, 16, 64), 200),
    ((16, 130, 8, 64), 200),
    ((4, 8, 136, 64), 160),
    ((128, 64, 4, 64), 128),
    # the innermost mode from the transposed images: row tails (I_{d-1} = 200,
    # 130, 150), a contraction tail (J = 120), two inner-group modes
    ((24, 120, 200), 300),
    ((10, 128, 130), 256),
    ((64, 8, 8, 150), 200),
    # 64-column image tiles with small I_k, natural and transposed images
    ((20, 3, 120), 48),
    ((8, 512, 20), 64),
    # the innermost mode read MN-major from the natural images needs I_{d-1} a
    # multiple of 8; at 4 mod 8 it takes the transposed images (128- and
    # 256-column tiles) and the other modes the 3xTF32 kernels
    ((64, 64, 132), 100),
    ((64, 64, 132), 256),
]

# shapes whose modes run on the fp16-split tensor-core kernels (value-range tests)
H2_SHAPES = [((130, 40, 48), 300), ((40, 36, 128), 450), ((200, 96, 64), 300), ((24, 120, 200), 300)]

# shapes with a mode whose main kernel converts Y in place and stores the fp16
# images (tc_convert=1; it runs first in an all-modes call), and that mode:
# mode 0 (slab scales by output row) with two row tiles, a 2-row tail, a column
# tail (R = 200 of 256); mode 1 and mode 2 (slab scales carried by G) with row
# and column tails and a 4-way tensor; 128-column (R = 100) and 64-column tiles
CONVERT_SHAPES = [
    ((256, 64, 128), 256, 0),
    ((130, 40, 128), 256, 0),
    ((384, 16, 64), 200, 0),
    ((16, 256, 128), 256, 1),
    ((24, 200, 128), 230, 1),
    ((3, 4, 256, 128), 256, 2),
    ((256, 64, 128), 100, 0),
    ((192, 64, 128), 64, 0),
]
