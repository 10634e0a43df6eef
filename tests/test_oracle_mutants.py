"""Plant plausible mistakes in the oracle (CPU only) and check the pins catch each one.

A pin set that no planted mistake can get past is the evidence that the oracle
is pinned to something other than itself.
"""

import types

import numpy as np
import pytest

import oracle
import oracle.collectives as oc
import pins

PUBLIC = [
    "bf16_bits_to_f32", "f32_to_bf16_rne", "fold_sum", "all_reduce", "reduce_scatter",
    "reduce_scatter_v", "all_gather", "all_to_all", "all_gather_v", "all_to_all_v",
]


def _fold_descending(columns):
    acc = np.array(columns[-1], dtype=np.float32, copy=True)
    for col in reversed(columns[:-1]):
        acc = np.add(acc, col, dtype=np.float32)
    return acc


def _fold_drop_last(columns):
    return oc.__dict__["_orig_fold"](columns[:-1] if len(columns) > 1 else columns)


def _fold_from_zero(columns):
    acc = np.zeros_like(np.asarray(columns[0], dtype=np.float32))
    for col in columns:
        acc = np.add(acc, col, dtype=np.float32)
    return acc


def _fold_pairwise(columns):
    cols = [np.asarray(c, dtype=np.float32) for c in columns]
    while len(cols) > 1:
        nxt = [np.add(cols[i], cols[i + 1], dtype=np.float32) for i in range(0, len(cols) - 1, 2)]
        if len(cols) % 2:
            nxt.append(cols[-1])
        cols = nxt
    return cols[0].copy()


def _fold_f64(columns):
    acc = np.zeros_like(np.asarray(columns[0], dtype=np.float64))
    for col in columns:
        acc = acc + np.asarray(col, dtype=np.float64)
    return acc.astype(np.float32)


def _fold_sign_flip(columns):
    acc = np.array(columns[0], dtype=np.float32, copy=True)
    for col in columns[1:-1]:
        acc = np.add(acc, col, dtype=np.float32)
    if len(columns) > 1:
        acc = np.subtract(acc, columns[-1], dtype=np.float32)
    return acc


def _bf16_truncate(x):
    u = np.asarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    return (u >> 16).astype(np.uint16).reshape(np.shape(x))


def _bf16_ties_away(x):
    u = np.asarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    return ((u + np.uint32(0x8000)) >> 16).astype(np.uint16).reshape(np.shape(x))


def _a2a_identity(inputs):
    return [np.array(b, copy=True) for b in inputs]


def _a2a_wrong_slot(inputs):
    world, n = len(inputs), inputs[0].size
    c = n // world
    out = []
    for d in range(world):
        dst = np.empty(n, dtype=inputs[0].dtype)
        for s in range(world):
            dst[s * c:(s + 1) * c] = inputs[s][s * c:(s + 1) * c]   # sends own chunk s, not chunk d
        out.append(dst)
    return out


def _rs_reversed(inputs, dtype):
    return list(reversed(oc.__dict__["_orig_rs"](inputs, dtype)))


def _ag_reversed(inputs):
    return oc.__dict__["_orig_ag"](list(reversed(inputs)))


def _agv_ignores_counts(inputs, counts):
    return oc.__dict__["_orig_ag"](inputs) if len({b.size for b in inputs}) == 1 else oc.__dict__["_orig_agv"](inputs, counts)


def _a2av_send_displ_wrong(inputs, counts):
    world = len(inputs)
    C = [[int(v) for v in row] for row in counts]
    out = []
    for d in range(world):
        dst = np.empty(sum(C[s][d] for s in range(world)), dtype=inputs[0].dtype)
        recv = 0
        for s in range(world):
            send = sum(C[k][d] for k in range(s))         # receive-side displacement used to send
            dst[recv:recv + C[s][d]] = inputs[s][send:send + C[s][d]]
            recv += C[s][d]
        out.append(dst)
    return out


MUTANTS = {
    "fold_descending": {"fold_sum": _fold_descending},
    "fold_drops_last_rank": {"fold_sum": _fold_drop_last},
    "fold_from_positive_zero": {"fold_sum": _fold_from_zero},
    "fold_pairwise_tree": {"fold_sum": _fold_pairwise},
    "fold_in_float64": {"fold_sum": _fold_f64},
    "fold_sign_flip": {"fold_sum": _fold_sign_flip},
    "bf16_truncates": {"f32_to_bf16_rne": _bf16_truncate},
    "bf16_ties_away": {"f32_to_bf16_rne": _bf16_ties_away},
    "a2a_identity": {"all_to_all": _a2a_identity},
    "a2a_wrong_slot": {"all_to_all": _a2a_wrong_slot},
    "rs_reversed_ranks": {"reduce_scatter": _rs_reversed},
    "ag_reversed_ranks": {"all_gather": _ag_reversed},
    "agv_ignores_counts": {"all_gather_v": _agv_ignores_counts},
    "a2av_wrong_send_displacement": {"all_to_all_v": _a2av_send_displ_wrong},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    monkeypatch.setitem(oc.__dict__, "_orig_fold", oc.fold_sum)
    monkeypatch.setitem(oc.__dict__, "_orig_rs", oc.reduce_scatter)
    monkeypatch.setitem(oc.__dict__, "_orig_ag", oc.all_gather)
    monkeypatch.setitem(oc.__dict__, "_orig_agv", oc.all_gather_v)
    ns = types.SimpleNamespace(**{k: getattr(oc, k) for k in PUBLIC})
    for k, fn in MUTANTS[name].items():
        monkeypatch.setattr(oc, k, fn)     # internal calls go through the module globals
        setattr(ns, k, fn)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(ns)
        except (AssertionError, ValueError, IndexError, TypeError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"


def test_real_oracle_passes_through_namespace():
    ns = types.SimpleNamespace(**{k: getattr(oc, k) for k in PUBLIC})
    for pin in pins.ALL_PINS:
        pin(ns)
