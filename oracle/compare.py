"""Parity bar between a GPU result and the oracle (test infrastructure only).

The bar, per output kind:
  * which cache bytes are written, every untouched byte, every UE8M0 scale byte
    and the pad byte: bit-exact;
  * E4M3 payload bytes: bit-exact except at most 1e-4 of them, and those at most
    one E4M3 step away (fp32 vs fp64 evaluation can sit on opposite sides of a
    rounding midpoint);
  * bf16 values (q, the 64 rope dims of an FP8 row, bf16 cache rows): within one
    bf16 ulp (adjacent representable values; +0 and -0 count as equal).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FP8_MISMATCH_BUDGET = 1e-4


def _ord_bf16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _ord_e4m3(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


@dataclass
class Report:
    ok: bool = True
    notes: list = field(default_factory=list)
    q_elems: int = 0
    q_ulp1: int = 0
    fp8_elems: int = 0
    fp8_step1: int = 0
    q_rows: int = 0  # q head rows compared (set by the caller that compares q)

    def fail(self, msg: str):
        self.ok = False
        self.notes.append(msg)

    def __str__(self):
        return (f"ok={self.ok} q: {self.q_ulp1}/{self.q_elems} at 1 ulp; fp8 payload: "
                f"{self.fp8_step1}/{self.fp8_elems} one step off; " + "; ".join(self.notes))


def compare_bf16(got: np.ndarray, ref: np.ndarray, what: str, rep: Report) -> Report:
    got = np.ascontiguousarray(got).view(np.uint16).ravel()
    ref = np.ascontiguousarray(ref).view(np.uint16).ravel()
    if got.shape != ref.shape:
        rep.fail(f"{what}: shape {got.shape} vs {ref.shape}")
        return rep
    d = np.abs(_ord_bf16(got) - _ord_bf16(ref))
    bad = np.nonzero(d > 1)[0]
    rep.q_elems += got.size
    rep.q_ulp1 += int((d == 1).sum())
    if bad.size:
        i = int(bad[0])
        rep.fail(f"{what}: {bad.size} bf16 values beyond 1 ulp, first at {i}: "
                 f"got {got[i]:#06x} want {ref[i]:#06x}")
    return rep


def written_slots(slots: np.ndarray, positions: np.ndarray, max_position: int,
                  num_slots: int) -> np.ndarray:
    """Mask of the cache slots a step writes: the slot of every token whose slot is in
    the cache and whose position is inside the cos/sin table.  A token with an
    out-of-range position writes nothing, so its slot must keep its old bytes."""
    slots = np.asarray(slots, np.int64)
    positions = np.asarray(positions, np.int64)
    ok = (slots >= 0) & (slots < num_slots) & (positions >= 0) & (positions < max_position)
    written = np.zeros(num_slots, dtype=bool)
    written[slots[ok]] = True
    return written


def compare_fp8_cache(got: np.ndarray, ref: np.ndarray, poison: np.ndarray, slots: np.ndarray,
                      positions: np.ndarray, max_position: int, num_blocks: int,
                      block_size: int, rep: Report) -> Report:
    """Compare two FP8 cache images (uint8, num_blocks*block_size*584 bytes);
    slots and positions are the step's per-token inputs."""
    got = np.ascontiguousarray(got).view(np.uint8).ravel()
    ref = np.ascontiguousarray(ref).view(np.uint8).ravel()
    nbs = block_size
    blocks = got[: num_blocks * nbs * 584].reshape(num_blocks, nbs * 584)
    rblocks = ref[: num_blocks * nbs * 584].reshape(num_blocks, nbs * 584)
    g_data = blocks[:, : nbs * 576].reshape(num_blocks * nbs, 576)
    r_data = rblocks[:, : nbs * 576].reshape(num_blocks * nbs, 576)
    g_scale = blocks[:, nbs * 576:].reshape(num_blocks * nbs, 8)
    r_scale = rblocks[:, nbs * 576:].reshape(num_blocks * nbs, 8)

    written = written_slots(slots, positions, max_position, num_blocks * nbs)
    # untouched slots: every byte equals the poison (and the oracle's image)
    pb = poison.reshape(num_blocks, nbs * 584)
    p_data = pb[:, : nbs * 576].reshape(num_blocks * nbs, 576)
    p_scale = pb[:, nbs * 576:].reshape(num_blocks * nbs, 8)
    un = ~written
    if not (np.array_equal(g_data[un], p_data[un]) and np.array_equal(g_scale[un], p_scale[un])):
        rep.fail("bytes of unwritten slots changed")
    if not (np.array_equal(r_data[un], p_data[un]) and np.array_equal(r_scale[un], p_scale[un])):
        rep.fail("oracle changed bytes of unwritten slots")
    # scale bytes + pad: exact
    gs, rs = g_scale[written], r_scale[written]
    if not np.array_equal(gs, rs):
        bad = np.nonzero((gs != rs).any(axis=1))[0]
        rep.fail(f"UE8M0 scale bytes differ in {bad.size} rows, first row {int(bad[0])}: "
                 f"got {gs[bad[0]].tolist()} want {rs[bad[0]].tolist()}")
    # payload: <= 1e-4 mismatches, each one step
    gp, rp = g_data[written, :448], r_data[written, :448]
    d = np.abs(_ord_e4m3(gp) - _ord_e4m3(rp))
    rep.fp8_elems += gp.size
    rep.fp8_step1 += int((d == 1).sum())
    if (d > 1).any():
        rep.fail(f"{int((d > 1).sum())} E4M3 payload bytes more than one step off")
    if gp.size and (d != 0).sum() > FP8_MISMATCH_BUDGET * gp.size:
        rep.fail(f"{int((d != 0).sum())} of {gp.size} E4M3 payload bytes differ (> 1e-4)")
    # rope tail: bf16 within one ulp
    compare_bf16(g_data[written, 448:].copy().view(np.uint16), r_data[written, 448:].copy().view(np.uint16),
                 "fp8-row rope dims", rep)
    return rep


def compare_bf16_cache(got: np.ndarray, ref: np.ndarray, poison: np.ndarray, slots: np.ndarray,
                       positions: np.ndarray, max_position: int, num_slots: int,
                       rep: Report) -> Report:
    g = np.ascontiguousarray(got).view(np.uint16).reshape(num_slots, 512)
    r = np.ascontiguousarray(ref).view(np.uint16).reshape(num_slots, 512)
    p = np.ascontiguousarray(poison).view(np.uint16).reshape(num_slots, 512)
    written = written_slots(slots, positions, max_position, num_slots)
    if not np.array_equal(g[~written], p[~written]):
        rep.fail("bytes of unwritten bf16 slots changed")
    if not np.array_equal(r[~written], p[~written]):
        rep.fail("oracle changed bytes of unwritten bf16 slots")
    compare_bf16(g[written], r[written], "bf16 cache rows", rep)
    return rep
