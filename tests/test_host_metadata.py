"""The library's host metadata builder (pkv_build_metadata) on CPU.

Pinned to the flatten example the "Model execution" page prints and its
exercise (tests/golden), compared with the Python runner builder and the
oracle's flatten on random schedules, and checked to reject inconsistent
schedules before writing anything.
"""

import ctypes
import json
import os
from types import SimpleNamespace

import numpy as np
import pytest

import workloads
from oracle import flatten as oracle_flatten
from paged_kv_attention_17_gb300 import build as pkv_build
from paged_kv_attention_17_gb300 import metadata


@pytest.fixture(scope="module")
def pkv():
    pkv_build.build()
    import paged_kv_attention_17_gb300 as p
    p.lib()
    return p


def _req(c, s, b):
    return SimpleNamespace(computed=c, scheduled=s, blocks=list(b))


def test_printed_example(pkv, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_example.json")))
    reqs = [_req(r["computed"], r["scheduled"], r["blocks"]) for r in g["schedule"]]
    m = metadata.build_native(reqs, g["block_size"])
    p = g["printed"]
    assert m["slot_mapping"].tolist() == p["slot_mapping"]
    assert m["query_start_loc"].tolist() == p["query_start_loc"]
    assert m["seq_lens"].tolist() == p["seq_lens"]
    assert m["positions"].tolist() == p["positions"]


def test_exercise(pkv, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_exercise.json")))
    r = g["request"]
    m = metadata.build_native([_req(r["computed"], r["scheduled"], r["blocks"])], g["block_size"])
    assert m["slot_mapping"].tolist() == g["expected"]["slot_mapping"]


@pytest.mark.parametrize("seed", range(12))
def test_matches_python_builder_and_oracle(pkv, seed):
    w = workloads.random_small(seed, num_seqs=11)
    a = metadata.build_native(w.requests)
    b = metadata.build(w.requests)
    o = oracle_flatten.flatten(w.requests)
    for k in ("query_start_loc", "seq_lens", "block_table", "slot_mapping", "positions"):
        assert a[k].tolist() == b[k].tolist(), k
    for k in ("query_start_loc", "seq_lens", "slot_mapping"):
        assert a[k].tolist() == o[k].tolist(), k
    for k in ("num_tokens", "max_query_len", "max_seq_len"):
        assert a[k] == b[k], k


def _call(pkv, computed, scheduled, offsets, ids, width, num_tokens):
    n = len(computed)
    arr = lambda x, t: np.ascontiguousarray(x, dtype=t)  # noqa: E731
    c, s, o, i = (arr(computed, np.int32), arr(scheduled, np.int32), arr(offsets, np.int32),
                  arr(ids, np.int32))
    qsl = np.full(n + 1, -7, dtype=np.int32)
    sl = np.full(n, -7, dtype=np.int32)
    tb = np.full((n, width), -7, dtype=np.int32)
    slots = np.full(max(num_tokens, 1), -7, dtype=np.int64)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)  # noqa: E731
    code = pkv.lib().pkv_build_metadata(n, p(c), p(s), p(o), p(i), 16, width, num_tokens, p(qsl),
                                        p(sl), p(tb), p(slots), None, None, None)
    return code, qsl, sl, tb, slots


def test_rejects_inconsistent_schedules_without_writing(pkv):
    ok = _call(pkv, [20, 0], [2, 3], [0, 2, 3], [5, 9, 4], 2, 5)
    assert ok[0] == 0 and ok[4].tolist() == [148, 149, 64, 65, 66]   # block 9 holds 16..31
    bad = [
        ([20, 0], [2, 3], [0, 1, 2], [5, 4], 2, 5),          # 22 tokens on one block
        ([20, 0], [2, 3], [0, 2, 3], [5, 9, 4], 2, 6),       # num_tokens != sum
        ([20, 0], [2, 3], [0, 2, 3], [5, -1, 4], 2, 5),      # negative block id
        ([20, 0], [2, 3], [0, 2, 3], [5, 9, 4], 1, 5),       # table too narrow
        ([-1, 0], [2, 3], [0, 2, 3], [5, 9, 4], 2, 5),       # negative count
        ([20, 0], [2, 3], [1, 2, 3], [5, 9, 4], 2, 5),       # offsets not starting at 0
    ]
    for args in bad:
        code, qsl, sl, tb, slots = _call(pkv, *args)
        assert code == 1, args
        assert (qsl == -7).all() and (sl == -7).all() and (tb == -7).all() and (slots == -7).all()
