"""The swizzled shared-memory image of a staged tile, looked at directly.

tsx_debug_stage_image (include/tsx_debug.h) loads one tile through a plan's
TMA loads into a cleared slot and copies the slot's raw bytes out.  The
image must be the tile's boxes placed one after another in the plan's slot,
each box's row-major bytes moved by ``oracle.structure.swizzle`` (CUDA's
definition of the 32/64/128-byte modes; TVM docs "copy_async -> tma",
"Demonstration program", names the 128-byte mode), with zeros where the box
reaches past the tensor or no box is loaded.  For the 8x256 fp16 tile of
that page the four rank-2 boxes and the one rank-3 box must leave
byte-identical images.
"""

import numpy as np
import pytest

from oracle import structure as st
from tests import _gpu
from tests._gpu import NP_BITS, random_bits, to_dev, torch

pytestmark = pytest.mark.gpu

ES = {"f16": 2, "bf16": 2, "f32": 4}
SWIZZLE_BYTES = {0: 0, 1: 32, 2: 64, 3: 128}


@pytest.fixture(scope="module")
def tsx():
    _gpu.need_gpu()
    import pipelined_elementwise_streaming_gb300 as m

    return m


def expected_image(bits: np.ndarray, info: dict, tile: int) -> np.ndarray:
    """The slot image the model predicts for tile `tile` of `bits`."""
    rows, cols = bits.shape
    es = info["elem_size"]
    rpl, chunks, atoms = info["rows_per_load"], info["row_chunks"], info["atoms"]
    inner, inner_bytes = info["inner_elems"], info["inner_bytes"]
    rank3 = info["rank"] == 3
    load_smem = info["slot_bytes"] // info["loads_per_operand"]
    swz = SWIZZLE_BYTES[info["swizzle"]]
    row0, col0 = st.tile_origin(tile, rows, cols, info["box_rows"], info["box_cols"])
    img = np.zeros(info["slot_bytes"], dtype=np.uint8)
    for r in range(chunks):
        r0 = row0 + r * rpl
        if r0 >= rows:
            continue                      # a box wholly below the tensor is not loaded
        for a in range(atoms):
            c0 = col0 + a * inner
            if c0 >= cols:
                continue                  # nor one wholly to its right
            box = np.zeros((rpl, inner), dtype=bits.dtype)
            part = bits[r0:r0 + rpl, c0:c0 + inner]
            box[:part.shape[0], :part.shape[1]] = part     # the rest reads as zero
            raw = box.view(np.uint8).reshape(-1)
            if rank3:
                load, first = r, a * rpl * inner_bytes     # atoms follow one another in one box
            else:
                load, first = r * atoms + a, 0
            for o in range(0, raw.size, 16):
                dst = load * load_smem + st.swizzle(first + o, swz)
                img[dst:dst + 16] = raw[o:o + 16]
    return img


CASES = [
    # dtype, rows, cols, box, stages, variant: swizzle mode, loads, edges
    ("f16", 8, 256, (8, 256), 1, "tma"),              # the page's tile: four 8x64 boxes, 128-byte swizzle
    ("f16", 8, 256, (8, 256), 1, "tma_rank3"),        # the same as one rank-3 box
    ("f32", 40, 1000, (8, 128), 4, "tma"),            # four 8x32 boxes; last column tile ragged
    ("f32", 40, 1024, (8, 128), 4, "tma_rank3"),
    ("bf16", 300, 520, (128, 128), 3, "tma"),         # two 128x64 boxes; ragged rows and columns
    ("f16", 50, 96, (16, 32), 2, "tma"),              # 64-byte rows: 64-byte swizzle
    ("f32", 20, 40, (8, 8), 2, "tma"),                # 32-byte rows: 32-byte swizzle
    ("f32", 16, 36, (8, 4), 2, "tma"),                # 16-byte rows: no swizzle
    ("f32", 600, 64, (512, 32), 1, "tma"),            # 512 rows: two row chunks of 256
    ("bf16", 64, 1000, (8, 512), 2, "tma_promoted"),  # one widened, unswizzled box per row chunk
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_staged_image_matches_the_swizzle_model(tsx, case):
    dtype, rows, cols, box, stages, variant = CASES[case]
    bits = random_bits(dtype, (rows, cols), 900 + case).view(NP_BITS[dtype])
    a = to_dev(bits, dtype)
    with tsx.Plan(dtype, rows, cols, box=box, stages=stages, variant=variant) as plan:
        info = plan.info("copy")
        tiles = info["tiles"]
        for tile in sorted({0, 1 % tiles, tiles // 2, tiles - 1}):
            got = plan.stage_image(a, tile).cpu().numpy()
            torch.cuda.synchronize()
            assert plan.status() == tsx.TSX_OK
            want = expected_image(bits, info, tile)
            bad = np.flatnonzero(got != want)
            assert bad.size == 0, (f"{variant} {dtype} box {box} tile {tile}: {bad.size} bytes differ, "
                                   f"first at {bad[0]}")


@pytest.mark.parametrize("dtype,rows,cols,box", [("f16", 8, 256, (8, 256)), ("f32", 40, 1024, (8, 128)),
                                                 ("bf16", 256, 512, (128, 128))])
def test_rank2_boxes_and_the_rank3_box_stage_the_same_bytes(tsx, dtype, rows, cols, box):
    bits = random_bits(dtype, (rows, cols), 77).view(NP_BITS[dtype])
    a = to_dev(bits, dtype)
    images = {}
    for variant in ("tma", "tma_rank3"):
        with tsx.Plan(dtype, rows, cols, box=box, stages=1, variant=variant) as plan:
            n = plan.info("copy")["tiles"]
            images[variant] = [plan.stage_image(a, t).cpu().numpy() for t in range(min(n, 6))]
            assert plan.status() == tsx.TSX_OK
    for x, y in zip(images["tma"], images["tma_rank3"]):
        assert np.array_equal(x, y)


def test_stage_image_declines(tsx):
    a = torch.zeros(64, 64, device="cuda")
    with tsx.Plan("f32", 64, 64, box=(8, 32), stages=2, variant="ldgsts") as plan:
        with pytest.raises(tsx.TsxError) as ei:
            plan.stage_image(a, 0)
        assert ei.value.code == tsx.TSX_ERR_UNSUPPORTED
    with tsx.Plan("f32", 64, 64, box=(8, 32), stages=2) as plan:
        with pytest.raises(tsx.TsxError) as ei:
            plan.stage_image(a, 16)
        assert ei.value.code == tsx.TSX_ERR_INVALID
