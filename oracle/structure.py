"""Integer plans the pages fix, written out plainly -- TEST INFRASTRUCTURE.

These are reference models for the host planner and the kernels' loop
structure; the library has its own implementation and never imports this.

* ``partition``   -- the ``[outer, threads, vec]`` split of a region
  (TVM docs "elementwise -> smem", section "Algorithm", step 2, and
  "copy_async -> ldgsts", section "Algorithm", step 1 with the table under
  "How inputs change the algorithm").
* ``split``       -- a stage tile cut into TMA boxes: every box dimension at
  most 256 and the innermost box inside the swizzle atom, several loads per
  stage, expect_tx = bytes per load x loads (nvFuser PR #2833 "Add TMA
  support for circular buffering pass", section "Lowering Details"; TVM docs
  "copy_async -> tma", table under "What it accepts" and "Algorithm" step 2).
* ``encode_args`` -- the ``cuTensorMapEncodeTiled`` argument list in the
  order the TVM page emits it ("copy_async -> tma", "Algorithm" step 3 and
  "Generated TIRx IR").
* ``swizzle``     -- where a byte of a box lands in shared memory under the
  32/64/128-byte swizzle modes (CUDA's definition; the pages name the mode
  only: parity unpinned beyond its invariants).
* ``schedule``    -- the pre-prologue / prologue / main / epilogue /
  post-epilogue event sequence of an S-stage circular buffer (nvFuser PR
  #2833, "Loop Structure" and "Detailed Pseudo-Code").
"""

from __future__ import annotations

from dataclasses import dataclass

ELEM_SIZE = {"f16": 2, "bf16": 2, "f32": 4}
DTYPE_NAME = {"f16": "float16", "bf16": "bfloat16", "f32": "float32"}
BOX_MAX = 256            # per box dimension (nvFuser PR #2833, "Lowering Details")
SWIZZLE_ATOM = 128       # bytes of the 128-B swizzle atom (TVM "copy_async -> tma")
SWIZZLE_CODE = {0: 0, 32: 1, 64: 2, 128: 3}   # CU_TENSOR_MAP_SWIZZLE_{NONE,32B,64B,128B}
L2_PROMO_128B = 2        # the value the TVM page passes
OOB_FILL_NONE = 0        # out-of-bounds elements read as zero


# --------------------------------------------------------------------------
# [outer, threads, vec]
# --------------------------------------------------------------------------

def partition(elems: int, threads: int, es: int, run_bytes: int, align_bytes: int,
              vec_bits=(128, 64, 32, 16)):
    """Widest vector that fits, then the round count.

    ``vec`` is the widest candidate width (in bits, from ``vec_bits``, widest
    first) that holds whole elements, divides the innermost contiguous run
    (``run_bytes``) and the guaranteed alignment (``align_bytes``), and for
    which ``threads * vec`` divides the region; ``outer = elems / (threads *
    vec)``.  Element ``v`` of round ``f`` of thread ``tid`` is the linear
    element ``(f * threads + tid) * vec + v``.  Returns ``(vec, outer)`` in
    elements, or ``None`` when no candidate fits (the variant declines).
    """
    for bits in sorted(vec_bits, reverse=True):
        vb = bits // 8
        if vb < es or vb % es:
            continue
        vec = vb // es
        if run_bytes % vb or align_bytes % vb:
            continue
        if elems % (threads * vec):
            continue
        return vec, elems // (threads * vec)
    return None


def linear_element(f: int, tid: int, v: int, threads: int, vec: int) -> int:
    return (f * threads + tid) * vec + v


LDGSTS_VEC_BITS = (128, 64, 32)   # cp.async copies 16, 8 or 4 bytes


# --------------------------------------------------------------------------
# Box split and expect_tx
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Split:
    mode: str                 # "rank2": one box per (row chunk, atom); "rank3": atoms as a 3rd dim
    inner_elems: int          # innermost box extent (elements)
    inner_bytes: int
    atoms: int                # lc: innermost boxes side by side along a tile row
    rows_per_load: int
    row_chunks: int           # lr: boxes stacked along rows
    loads_per_operand: int
    bytes_per_load: int
    swizzle_bytes: int        # 128 / 64 / 32, or 0 for none

    def tx_bytes(self, n_in: int) -> int:
        """expect_tx of one stage: bytes per load x loads per stage."""
        return n_in * self.loads_per_operand * self.bytes_per_load


def split(dtype: str, box_rows: int, box_cols: int, mode: str = "rank2", cols: int | None = None):
    """Cut a ``box_rows x box_cols`` stage tile into TMA boxes.

    Returns a ``Split``, or ``None`` when no legal descriptor exists (the
    variant declines): a zero extent, a tile row that is not a whole number
    of 16-byte units, a row wider than one atom that is not a whole number
    of atoms, or rows that cannot be cut into equal chunks of at most 256.
    The rank-3 form also needs the tensor's row length ``cols`` to be a
    whole number of atoms, because the atom axis walks along the row.
    """
    es = ELEM_SIZE[dtype]
    if box_rows <= 0 or box_cols <= 0:
        return None
    row_bytes = box_cols * es
    if row_bytes % 16:
        return None
    inner_bytes = min(row_bytes, SWIZZLE_ATOM)
    if row_bytes % inner_bytes:
        return None
    inner_elems = inner_bytes // es
    atoms = row_bytes // inner_bytes
    row_chunks = -(-box_rows // BOX_MAX)
    if box_rows % row_chunks:
        return None
    rows_per_load = box_rows // row_chunks
    swz = inner_bytes if inner_bytes in (32, 64, 128) else 0
    if mode == "rank2":
        return Split(mode, inner_elems, inner_bytes, atoms, rows_per_load, row_chunks,
                     atoms * row_chunks, rows_per_load * inner_bytes, swz)
    if mode == "rank3":
        if cols is None or cols % inner_elems or atoms > BOX_MAX:
            return None
        return Split(mode, inner_elems, inner_bytes, atoms, rows_per_load, row_chunks,
                     row_chunks, rows_per_load * inner_bytes * atoms, swz)
    raise ValueError(mode)


PROMOTION_CHAIN = (1, 2, 4, 8)   # element sizes a descriptor may be widened to


def promote(es: int, row_bytes: int, cols_bytes: int):
    """Element size for a box that spans a whole tile row without a swizzle.

    TVM docs "copy_async -> tma", table under "How inputs change the
    algorithm": a box of more than 256 elements triggers element-type
    promotion along 1 -> 2 -> 4 -> 8 bytes.  The smallest size of the chain,
    at least the element's own, that holds the row in at most 256 elements
    and divides both the tile row and the tensor row; None when even 8
    bytes cannot (the variant declines).
    """
    for pes in PROMOTION_CHAIN:
        if pes < es or row_bytes % pes or cols_bytes % pes:
            continue
        if row_bytes // pes <= BOX_MAX:
            return pes
    return None


def encode_args(dtype: str, rows: int, cols: int, sp: Split) -> tuple:
    """The tiled-encode argument list, in the TVM page's order.

    ``(dtype, rank, *reversed(shape), *reversed(strides[:-1]),
    *reversed(box), *element_strides, interleave, swizzle, l2_promotion,
    oob_fill)`` with strides in bytes.  Rank 2 views the tensor as
    ``[rows, cols]``; rank 3 as ``[cols / atom, rows, atom]`` with the atom
    axis striding by one atom's bytes.
    """
    es = ELEM_SIZE[dtype]
    if sp.mode == "rank2":
        shape = (rows, cols)
        strides = (cols * es, es)
        box = (sp.rows_per_load, sp.inner_elems)
    else:
        shape = (cols // sp.inner_elems, rows, sp.inner_elems)
        strides = (sp.inner_bytes, cols * es, es)
        box = (sp.atoms, sp.rows_per_load, sp.inner_elems)
    rank = len(shape)
    return (DTYPE_NAME[dtype], rank, *reversed(shape), *reversed(strides[:-1]), *reversed(box),
            *([1] * rank), 0, SWIZZLE_CODE[sp.swizzle_bytes], L2_PROMO_128B, OOB_FILL_NONE)


# --------------------------------------------------------------------------
# The swizzled shared-memory layout of a box
# --------------------------------------------------------------------------

def swizzle(offset: int, swizzle_bytes: int) -> int:
    """Shared-memory byte offset, within a box that starts on a 1024-byte
    boundary, of the byte at row-major offset ``offset`` of the box.

    The pages name the 128-byte swizzle of TMA loads (TVM docs
    "copy_async -> tma", "Demonstration program") but print no swizzled
    address, so this follows CUDA's documented definition of the tensor-map
    swizzle modes: the 16-byte chunk index (address bits 4..6) is XOR-ed
    with the 128-byte line index (bits 7..9), keeping three bits for the
    128-byte mode, two for the 64-byte mode and one for the 32-byte mode;
    mode 0 leaves the layout row-major.  Parity unpinned against the pages:
    only its invariants (a permutation of whole 16-byte chunks within each
    period, its own inverse, line 0 fixed) are checked on the CPU.
    """
    bits = {0: 0, 32: 1, 64: 2, 128: 3}[swizzle_bytes]
    if not bits:
        return offset
    mask = (1 << bits) - 1
    return offset ^ (((offset >> 7) & mask) << 4)


# --------------------------------------------------------------------------
# Tiles, persistent assignment and the S-stage schedule
# --------------------------------------------------------------------------

def tile_count(rows: int, cols: int, box_rows: int, box_cols: int) -> int:
    return (-(-rows // box_rows)) * (-(-cols // box_cols))


def tile_origin(t: int, rows: int, cols: int, box_rows: int, box_cols: int):
    """Row-major tile order: (row0, col0) of tile ``t``."""
    tiles_c = -(-cols // box_cols)
    return (t // tiles_c) * box_rows, (t % tiles_c) * box_cols


def cta_tiles(T: int, G: int, cta: int) -> list:
    """A persistent CTA ``cta`` of ``G`` takes tiles cta, cta + G, ..."""
    return list(range(cta, T, G))


def schedule(N: int, S: int) -> list:
    """Event list of one CTA streaming ``N`` tiles through ``S`` stages.

    Events: ("init", s), ("load", k, stage), ("wait", k, stage, parity),
    ("body", k), ("inval", s).  The prologue issues the first S - 1 loads,
    the main loop runs N - (S - 1) iterations that each issue the load for
    tile i + S - 1 into stage (i + S - 1) mod S and then wait on tile i, the
    epilogue waits on the remaining tiles; parity of the k-th use of a stage
    is (k / S) mod 2.  Ranges that would be negative for N < S - 1 are empty.
    """
    ev = [("init", s) for s in range(S)]
    for k in range(min(S - 1, N)):
        ev.append(("load", k, k % S))
    main = max(0, N - (S - 1))
    for i in range(main):
        k = i + S - 1
        ev.append(("load", k, k % S))
        ev.append(("wait", i, i % S, (i // S) & 1))
        ev.append(("body", i))
    for i in range(main, N):
        ev.append(("wait", i, i % S, (i // S) & 1))
        ev.append(("body", i))
    ev.extend(("inval", s) for s in range(S))
    return ev


def trip_counts(N: int, S: int):
    """(prologue loads, main iterations, epilogue iterations)."""
    main = max(0, N - (S - 1))
    return min(S - 1, N), main, N - main


def ldgsts_pending_allowed(i: int, N: int, S: int) -> int:
    """cp.async groups that may stay in flight when tile ``i`` is consumed.

    Groups are committed one per tile in tile order; before the issue of
    iteration i, tiles 0 .. min(N, i + S - 1) - 1 are committed, so waiting
    until at most ``min(N, i + S - 1) - i - 1`` groups are pending leaves
    tile i complete.  That is S - 2 in the main loop and N - 1 - i in the
    epilogue (S >= 2).
    """
    return min(N, i + S - 1) - i - 1
