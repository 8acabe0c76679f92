"""Helpers shared by the GPU parity tests: run the oracle on the same seeded inputs and
compare with the CUDA path (bit-exact for codes and scales, the stated tolerance for Y)."""

from typing import Optional, Sequence

import numpy as np
import torch

from oracle import fp8_oracle as O


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_weight(w: torch.Tensor, per_channel: bool, rows: Optional[np.ndarray] = None, fmt: str = "e4m3"):
    """Oracle qW/s_w for the selected rows (per-tensor scale from the full W)."""
    w32 = f32(w)
    sel = w32 if rows is None else w32[rows]
    if per_channel:
        return O.quantize_per_row(sel, fmt)
    s = np.float32(O.scale_from_amax(O.amax(w32), fmt))
    return O.quantize_with_scale(sel, s, fmt), s


def oracle_act(a: torch.Tensor, rows: Optional[np.ndarray] = None, fmt: str = "e4m3", s_static=None):
    """Oracle qA/s_a for the selected rows: dynamic scale from all of A, or the static one."""
    a32 = f32(a)
    s = np.float32(O.scale_from_amax(O.amax(a32), fmt)) if s_static is None else np.float32(s_static)
    sel = a32 if rows is None else a32[rows]
    return O.quantize_with_scale(sel, s, fmt), s


def assert_codes_equal(q_gpu: torch.Tensor, q_ref: np.ndarray, K: int, what: str):
    """Logical region bit-exact, padding bytes [K, ld) zero."""
    q = q_gpu.cpu().numpy()
    got = q[:, :K]
    bad = np.argwhere(got != q_ref)
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[:5].tolist()} " \
                          f"got {got[tuple(bad[:5].T)]} want {q_ref[tuple(bad[:5].T)]}"
    assert not np.any(q[:, K:]), f"{what}: padding bytes not zero"


def assert_scale_equal(s_gpu: torch.Tensor, s_ref, what: str):
    got = s_gpu.cpu().numpy().astype(np.float32)
    want = np.asarray(s_ref, np.float32).reshape(got.shape)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"{what}: scale {got[:4]} != {want[:4]}"


def assert_y_within_tolerance(y_gpu: np.ndarray, qa, s_a, qw, s_w, bias: Optional[np.ndarray], what: str,
                              fmt_a: str = "e4m3", fmt_w: str = "e4m3"):
    y_ref = O.scaled_mm(qa, s_a, qw, s_w, bias, fmt_a=fmt_a, fmt_w=fmt_w)
    tol = O.tolerance(qa, s_a, qw, s_w, y_ref, fmt_a, fmt_w)
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{what}: {len(bad)} of {err.size} outputs outside tolerance; first "
                           f"{bad[:3].tolist()} got {y_gpu[tuple(bad[:3].T)]} want {y_ref[tuple(bad[:3].T)]} "
                           f"tol {tol[tuple(bad[:3].T)]}")
    return float(np.max(err / tol)) if err.size else 0.0


def linear_parity(y: torch.Tensor, a: torch.Tensor, w: torch.Tensor, per_channel: bool,
                  bias: Optional[torch.Tensor] = None, rows: Optional[Sequence[int]] = None,
                  cols: Optional[Sequence[int]] = None, what: str = "Y", fmt_a: str = "e4m3",
                  fmt_w: str = "e4m3", s_static=None) -> float:
    """Compare the library's Y (full [M, N] on device) with the oracle on rows x cols."""
    rows = np.arange(a.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(w.shape[0]) if cols is None else np.asarray(cols)
    qa, s_a = oracle_act(a, rows, fmt_a, s_static)
    qw, s_w = oracle_weight(w, per_channel, cols, fmt_w)
    b = None if bias is None else f32(bias)[cols]
    y_gpu = f32(y)[np.ix_(rows, cols)]
    return assert_y_within_tolerance(y_gpu, qa, s_a, qw, s_w, b, what, fmt_a, fmt_w)


def guarded(shape, dtype, device, guard: int = 64, fill: int = 0x5A):
    """A tensor view inside a larger buffer whose guard bands hold a canary byte pattern."""
    rows, cols = shape
    elt = torch.tensor([], dtype=dtype).element_size()
    ld = cols + guard
    buf = torch.full(((rows + 2) * ld * elt + 2 * guard * elt,), fill, dtype=torch.uint8, device=device)
    base = ld * elt + guard * elt
    view = buf[base: base + rows * ld * elt].view(dtype).view(rows, ld)[:, :cols]
    return buf, view, base, ld * elt, cols * elt


def assert_guards_intact(buf: torch.Tensor, base: int, row_bytes: int, used: int, rows: int, fill: int = 0x5A):
    b = buf.cpu().numpy()
    mask = np.ones(b.size, bool)
    for r in range(rows):
        mask[base + r * row_bytes: base + r * row_bytes + used] = False
    assert np.all(b[mask] == fill), "write outside the output region"


def weight_only_parity(y: torch.Tensor, a: torch.Tensor, w: torch.Tensor, per_channel: bool,
                       bias: Optional[torch.Tensor] = None, rows: Optional[Sequence[int]] = None,
                       cols: Optional[Sequence[int]] = None, what: str = "Y", fmt_w: str = "e4m3") -> float:
    """Weight-only linear against the oracle (bf16 A, FP8 W quantized by the oracle) on rows x cols."""
    rows = np.arange(a.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(w.shape[0]) if cols is None else np.asarray(cols)
    a_sel = f32(a)[rows]
    qw, s_w = oracle_weight(w, per_channel, cols, fmt_w)
    b = None if bias is None else f32(bias)[cols]
    y_ref = O.linear_weight_only(a_sel, qw, s_w, b, fmt_w)
    tol = O.tolerance_weight_only(a_sel, qw, s_w, y_ref, fmt_w)
    y_gpu = f32(y)[np.ix_(rows, cols)]
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{what}: {len(bad)} of {err.size} outputs outside tolerance; first "
                           f"{bad[:3].tolist()} got {y_gpu[tuple(bad[:3].T)]} want {y_ref[tuple(bad[:3].T)]} "
                           f"tol {tol[tuple(bad[:3].T)]}")
    return float(np.max(err / tol)) if err.size else 0.0


def tail_split_expected(tiles: int, slots: int, largest: int) -> int:
    """Column split of a GEMM's last wave: the largest factor (4, 2, at most `largest`) whose
    units still fit one wave of `slots`; 1 when the tiles fill whole waves or fit one."""
    rem = tiles % slots
    if tiles <= slots or rem == 0:
        return 1
    return next((f for f in (4, 2) if f <= largest and f * rem <= slots), 1)


def tail_rows(n_tiles: int, slots: int, split: int, rows_per_unit: int) -> int:
    """Smallest M (ragged: short of a whole last unit) whose tile count leaves a last wave that
    splits into `split` units per tile on `slots` slots."""
    for units in range(2, 512):
        if tail_split_expected(units * n_tiles, slots, split) == split:
            return units * rows_per_unit - rows_per_unit // 3
    raise AssertionError("no such M")
