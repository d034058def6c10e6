"""Host logic of the CUDA-graph capture ladder (no GPU): the ladder and its
bucketing pinned to the page's printed padding table, the packed input layout,
and the padding of a step to its captured size."""

import json
import os

import torch

from paged_kv_attention_17_gb300.graphs import InputLayout, bucket, capture_ladder, fill_padding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "capture_ladder.json")


def test_capture_ladder_matches_page():
    g = json.load(open(GOLDEN))
    sizes = capture_ladder(512)
    assert len(sizes) == g["num_sizes"]
    assert sizes[:6] == g["first_sizes"] and sizes[-3:] == g["last_sizes"]
    for row in g["padding_table"]:
        got = bucket(row["tokens"], sizes)
        assert got == row["graph"], row
        if got is not None:
            assert got - row["tokens"] == row["padded"], row


def test_ladder_is_sorted_and_capped():
    for top in (1, 3, 8, 64, 100, 256, 512):
        s = capture_ladder(top)
        assert s == sorted(set(s)) and s[0] == 1 and s[-1] <= top


def test_input_layout_aligned_and_disjoint():
    for b in (1, 4, 64):
        lay = InputLayout.of(b, 32, 8, 128, 2, 512)
        spans = sorted(lay.offsets.values())
        assert all(off % 256 == 0 for off, _ in spans)
        for (o1, n1), (o2, _) in zip(spans, spans[1:]):
            assert o1 + n1 <= o2
        assert spans[-1][0] + spans[-1][1] <= lay.nbytes
        assert lay.offsets["q"][1] == b * 32 * 128 * 2
        assert lay.offsets["query_start_loc"][1] == (b + 1) * 4


def test_padding_rows_are_empty_requests():
    b, n = 8, 5
    qsl = torch.full((b + 1,), 99, dtype=torch.int32)
    slots = torch.full((b,), 7, dtype=torch.int64)
    lens = torch.full((b,), 9, dtype=torch.int32)
    table = torch.full((b, 4), 3, dtype=torch.int32)
    fill_padding(qsl, slots, lens, table, n, b)
    assert qsl.tolist() == [0, 1, 2, 3, 4, 5, 5, 5, 5]
    assert slots[n:].tolist() == [-1] * (b - n) and slots[:n].tolist() == [7] * n
    assert lens[n:].tolist() == [0] * (b - n) and lens[:n].tolist() == [9] * n
    assert int(table[n:].abs().sum()) == 0
