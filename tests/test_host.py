"""Host-side checks that need no GPU: the library builds, loads and exports
every symbol of include/pkv.h; the runner-side metadata builder reproduces the
page's printed flatten example and agrees with the oracle's builder; workspace
sizing and host validation return the documented statuses without enqueuing
anything."""

import ctypes
import json
import os
import re
from types import SimpleNamespace

import numpy as np
import pytest

import workloads
from oracle import flatten as oracle_flatten
from paged_kv_attention_17_gb300 import build as pkv_build
from paged_kv_attention_17_gb300 import metadata

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    pkv_build.build()
    import paged_kv_attention_17_gb300 as p
    p.lib()
    return p


def _header_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_header_symbol(pkv):
    names = _header_functions()
    assert names == sorted(pkv.EXPORTS)
    for n in names:
        assert hasattr(pkv.lib(), n), n


def test_status_strings(pkv):
    assert pkv.pkv_status_string(0) == "PKV_OK"
    assert pkv.pkv_status_string(3) == "PKV_ERR_WORKSPACE"
    assert pkv.pkv_status_string(99) == "PKV_UNKNOWN_STATUS"


def _req(c, s, b):
    return SimpleNamespace(computed=c, scheduled=s, blocks=list(b))


def test_metadata_matches_printed_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_example.json")))
    reqs = [_req(r["computed"], r["scheduled"], r["blocks"]) for r in g["schedule"]]
    m = metadata.build(reqs, g["block_size"])
    p = g["printed"]
    assert m["slot_mapping"].tolist() == p["slot_mapping"]
    assert m["query_start_loc"].tolist() == p["query_start_loc"]
    assert m["seq_lens"].tolist() == p["seq_lens"]
    assert m["positions"].tolist() == p["positions"]
    assert m["query_start_loc"].dtype == np.int32 and m["slot_mapping"].dtype == np.int64


def test_metadata_exercise(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_exercise.json")))
    r = g["request"]
    m = metadata.build([_req(r["computed"], r["scheduled"], r["blocks"])], g["block_size"])
    assert m["slot_mapping"].tolist() == g["expected"]["slot_mapping"]


@pytest.mark.parametrize("seed", range(6))
def test_metadata_agrees_with_oracle_builder(seed):
    w = workloads.random_small(seed, num_seqs=9)
    m = metadata.build(w.requests)
    o = oracle_flatten.flatten(w.requests)
    for k in ("slot_mapping", "query_start_loc", "seq_lens", "positions"):
        assert m[k].tolist() == o[k].tolist(), k
    ctx = metadata.context_slot_mapping(w.requests)
    want = np.concatenate([oracle_flatten.context_slots(r) for r in w.requests])
    assert ctx.tolist() == want.tolist()


def test_workspace_bytes(pkv):
    assert pkv.pkv_workspace_bytes(1, 32, 128, 1) == 0
    rows = 7 * 3 * 4 * 32
    want = -(-(rows * 128 * 4) // 256) * 256 + -(-(rows * 4) // 256) * 256
    assert pkv.pkv_workspace_bytes(3, 32, 128, 7) == want


def _attn_call(pkv, **over):
    L = pkv.lib()
    args = dict(q=16, k=16, v=16, out=16, lse=0, qsl=16, sl=16, bt=16, mbps=4, num_seqs=2,
                num_tokens=5, max_q=4, max_s=40, hq=8, hkv=2, d=128, bs=16, scale=0.1, causal=1,
                splits=1, ws=0, ws_bytes=0, flag=0, num_blocks=10, dtype=1, stream=0)
    args.update(over)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.pkv_attention_varlen(vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["out"]),
                                  vp(args["lse"]), vp(args["qsl"]), vp(args["sl"]), vp(args["bt"]),
                                  args["mbps"], args["num_seqs"], args["num_tokens"], args["max_q"],
                                  args["max_s"], args["hq"], args["hkv"], args["d"], args["bs"],
                                  args["scale"], args["causal"], args["splits"], vp(args["ws"]),
                                  args["ws_bytes"], vp(args["flag"]), args["num_blocks"],
                                  args["dtype"], vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(hq=6, hkv=4), 1),            # Hq not a multiple of Hkv
    (dict(d=96), 2),                   # unsupported head_dim
    (dict(bs=32), 2),                  # unsupported block size
    (dict(dtype=7), 1),                # unknown dtype
    (dict(q=0), 1),                    # null q
    (dict(q=24), 1),                   # misaligned q
    (dict(splits=65), 1),              # too many splits
    (dict(splits=4), 3),               # split partials need a workspace
    (dict(splits=4, ws=4096, ws_bytes=16), 3),
    (dict(max_q=0), 1),
    (dict(scale=float("nan")), 1),
    (dict(num_tokens=0), 0),           # empty batch: no-op
    (dict(num_seqs=0), 0),
    (dict(num_seqs=65536), 2),         # beyond the request grid
    (dict(num_blocks=1 << 27), 2),     # 2^31 slots: beyond int32 TMA coordinates
    (dict(mbps=2, max_s=33), 1),       # a 2-block table row holds at most 32 keys
])
def test_attention_host_validation(pkv, over, code):
    assert _attn_call(pkv, **over) == code


def test_stage_inputs_host_validation(pkv):
    L = pkv.lib()
    vp = ctypes.c_void_p
    # zero bytes is a no-op; sizes that are not whole 16-byte words, negative
    # sizes, null and misaligned pointers are rejected before any launch
    assert L.pkv_stage_inputs(None, None, 0, None) == 0
    assert L.pkv_stage_inputs(vp(16), vp(16), 24, None) == 1
    assert L.pkv_stage_inputs(vp(16), vp(16), -16, None) == 1
    assert L.pkv_stage_inputs(None, vp(16), 32, None) == 1
    assert L.pkv_stage_inputs(vp(16), None, 32, None) == 1
    assert L.pkv_stage_inputs(vp(24), vp(16), 32, None) == 1
    assert L.pkv_stage_inputs(vp(16), vp(40), 32, None) == 1


def test_e4m3_window_and_cascade_host_validation(pkv):
    # the E4M3 sliding-window and shared-prefix entry points reject bad scales
    # and a negative window before touching any pointer or launching
    L = pkv.lib()
    vp = ctypes.c_void_p
    win = lambda ks, vs, window: L.pkv_attention_varlen_e4m3_window(
        None, None, None, None, None, None, None, None, 4, 1, 1, 1, 64, 8, 2, 128, 16,
        0.1, ks, vs, 1, window, 0, None, 0, None, 4, None)
    assert win(0.0, 1.0, 0) == 1
    assert win(1.0, float("inf"), 0) == 1
    assert win(1.0, 1.0, -1) == 1
    casc = lambda ks, vs: L.pkv_cascade_attention_e4m3(
        None, None, None, None, None, None, None, None, 4, None, 0, 1, 1, 1, 64, 8, 2, 128, 16,
        0.1, ks, vs, 0, None, 0, None, 4, None)
    assert casc(-1.0, 1.0) == 1
    assert casc(1.0, float("nan")) == 1
    # valid scales: an empty batch is a no-op
    assert L.pkv_cascade_attention_e4m3(None, vp(16), vp(16), None, None, None, None, None, 4,
                                        None, 0, 0, 0, 1, 64, 8, 2, 128, 16, 0.1, 1.0, 1.0, 0,
                                        None, 0, None, 4, None) == 0


def test_write_host_validation(pkv):
    L = pkv.lib()
    vp = ctypes.c_void_p
    # empty batch is a no-op; bad sizes and null pointers are rejected
    assert L.pkv_write(None, None, None, 0, None, None, 4, 16, 8, 128, 1, None, None) == 0
    assert L.pkv_write(vp(16), vp(16), vp(16), 3, vp(16), vp(16), 4, 8, 8, 128, 1, None, None) == 2
    assert L.pkv_write(None, vp(16), vp(16), 3, vp(16), vp(16), 4, 16, 8, 128, 1, None, None) == 1
    assert L.pkv_write(vp(16), vp(16), vp(16), -1, vp(16), vp(16), 4, 16, 8, 128, 1, None, None) == 1
    assert L.pkv_write(vp(18), vp(16), vp(16), 3, vp(16), vp(16), 4, 16, 8, 128, 1, None, None) == 1


def _attn_e4m3_call(pkv, **over):
    L = pkv.lib()
    args = dict(q=16, k=16, v=16, out=16, lse=0, qsl=16, sl=16, bt=16, mbps=4, num_seqs=2,
                num_tokens=5, max_q=4, max_s=40, hq=8, hkv=2, d=128, bs=16, scale=0.1, ks=0.5,
                vs=0.25, causal=1, splits=1, ws=0, ws_bytes=0, flag=0, num_blocks=10, stream=0)
    args.update(over)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.pkv_attention_varlen_e4m3(
        vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["out"]), vp(args["lse"]),
        vp(args["qsl"]), vp(args["sl"]), vp(args["bt"]), args["mbps"], args["num_seqs"],
        args["num_tokens"], args["max_q"], args["max_s"], args["hq"], args["hkv"], args["d"],
        args["bs"], args["scale"], args["ks"], args["vs"], args["causal"], args["splits"],
        vp(args["ws"]), args["ws_bytes"], vp(args["flag"]), args["num_blocks"], vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(ks=0.0), 1),                 # scales must be finite and positive
    (dict(vs=-1.0), 1),
    (dict(ks=float("inf")), 1),
    (dict(vs=float("nan")), 1),
    (dict(d=96), 2),
    (dict(q=24), 1),
    (dict(splits=4), 3),
    (dict(num_tokens=0), 0),
])
def test_attention_e4m3_host_validation(pkv, over, code):
    assert _attn_e4m3_call(pkv, **over) == code


def test_write_e4m3_host_validation(pkv):
    L = pkv.lib()
    vp = ctypes.c_void_p
    ok = (4, 16, 8, 128, 1, 1.0, 1.0, None, None)
    assert L.pkv_write_e4m3(None, None, None, 0, None, None, *ok) == 0
    assert L.pkv_write_e4m3(vp(16), vp(16), vp(16), 3, vp(16), vp(16),
                            4, 16, 8, 128, 1, 0.0, 1.0, None, None) == 1
    assert L.pkv_write_e4m3(vp(16), vp(16), vp(16), 3, vp(16), vp(16),
                            4, 16, 8, 128, 1, 1.0, float("nan"), None, None) == 1
    assert L.pkv_write_e4m3(vp(16), vp(16), vp(16), 3, vp(16), vp(16),
                            4, 16, 8, 128, 5, 1.0, 1.0, None, None) == 1      # source dtype
    assert L.pkv_write_e4m3(vp(16), vp(16), vp(16), 3, vp(16), vp(16),
                            4, 16, 1, 8, 1, 1.0, 1.0, None, None) == 2        # row of 8 codes
    assert L.pkv_write_e4m3(vp(16), vp(16), vp(16), 3, vp(16), vp(24), *ok) == 1


def _cascade_call(pkv, **over):
    L = pkv.lib()
    args = dict(q=16, k=16, v=16, out=16, lse=0, qsl=16, sl=16, bt=16, mbps=4, shared=16,
                shared_blocks=3, num_seqs=2, num_tokens=2, max_q=1, max_s=40, hq=8, hkv=2, d=128,
                bs=16, scale=0.1, splits=2, ws=0, ws_bytes=0, flag=0, num_blocks=10, dtype=1,
                stream=0)
    args.update(over)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.pkv_cascade_attention(
        vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["out"]), vp(args["lse"]),
        vp(args["qsl"]), vp(args["sl"]), vp(args["bt"]), args["mbps"], vp(args["shared"]),
        args["shared_blocks"], args["num_seqs"], args["num_tokens"], args["max_q"], args["max_s"],
        args["hq"], args["hkv"], args["d"], args["bs"], args["scale"], args["splits"],
        vp(args["ws"]), args["ws_bytes"], vp(args["flag"]), args["num_blocks"], args["dtype"],
        vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(), 3),                       # no workspace for 2 prefix splits + own part
    (dict(ws=4096, ws_bytes=64), 3),
    (dict(splits=64), 1),              # at most 63 prefix splits
    (dict(splits=-1), 1),
    (dict(shared_blocks=-1), 1),
    (dict(shared=0), 1),               # shared blocks named but no table
    (dict(hq=6, hkv=4), 1),
    (dict(d=96), 2),
    (dict(bs=32), 2),
    (dict(dtype=7), 1),
    (dict(q=24), 1),
    (dict(num_tokens=0), 0),
    (dict(mbps=2, max_s=33, ws=4096, ws_bytes=1 << 20), 1),   # own keys beyond the table row
])
def test_cascade_host_validation(pkv, over, code):
    assert _cascade_call(pkv, **over) == code


def test_cascade_workspace_and_split_rule(pkv):
    rows = 3 * 5 * 8
    want = -(-(rows * 128 * 4) // 256) * 256 + -(-(rows * 4) // 256) * 256
    assert pkv.pkv_cascade_workspace_bytes(5, 8, 128, 2) == want
    L = pkv.lib()
    assert L.pkv_cascade_splits(5, 0, 8, 2, 128, 1, 0) == 0   # no prefix: no prefix pass
    assert L.pkv_cascade_splits(0, 4, 8, 2, 128, 1, 0) == -1
    assert L.pkv_cascade_splits(5, 4, 6, 4, 128, 1, 0) == -1
    assert L.pkv_cascade_splits(5, 4, 8, 2, 128, 7, 0) == -1  # unknown dtype


def test_num_splits_rejects_bad_args(pkv):
    assert pkv.lib().pkv_num_splits(0, 1, 100, 32, 8, 128, 0) == 0
    assert pkv.lib().pkv_num_splits(1, 1, 100, 30, 8, 128, 0) == 0
