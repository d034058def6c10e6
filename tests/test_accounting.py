"""The benchmark's algorithmic-work accounting, pinned to the pages' figures
and closed forms.

"Anatomy of a serving engine" (section "Capacity belongs to the KV cache
manager") gives 327,680 bytes of K/V per token for 80 layers x 8 KV heads x
head_dim 128 at 2 bytes; "Inside the engine ..." (section "Never materialise
the TxT matrix") gives 128 MB for one head's 8192 x 8192 fp16 score matrix.
The decode bytes count each KV head once over seq_len tokens; the prefill
FLOPs count 4 D H_q per visible (query, key) pair.
"""

from types import SimpleNamespace

import bench
import workloads


def _r(c, s):
    return SimpleNamespace(computed=c, scheduled=s)


def test_kv_bytes_per_token_of_the_70b_shape():
    assert 80 * bench.kv_bytes([_r(0, 1)], 8, 128, 2) == 327_680


def test_materialised_score_matrix_is_128_mib():
    assert 8192 * 8192 * 2 == 128 * 2 ** 20


def test_decode_8k_bytes():
    w = workloads.decode_8k()
    assert bench.kv_bytes(w.requests, 8, 128, 2) == 2 * 8192 * 8 * 128 * 2 == 33_554_432
    w8 = workloads.decode_8k_e4m3()
    assert bench.kv_bytes(w8.requests, 8, 128, 1) == 16_777_216


def test_prefill_8k_flops():
    w = workloads.prefill_8k()
    assert bench.causal_flops(w.requests, 32, 128) == 4 * 128 * 32 * (8192 * 8193 // 2)
    assert abs(bench.causal_flops(w.requests, 32, 128) - 5.498e11) < 0.001e11


def test_mixed_chunk_flops_and_tail():
    # the 2048-token chunk on an empty prefix: sum of (i + 1) visible keys
    assert bench.causal_flops([_r(0, 2048)], 32, 128) == 16384 * (2048 * 2049 // 2)
    # a 3-token tail on 1000 cached keys sees 1001, 1002, 1003 keys
    assert bench.causal_flops([_r(1000, 3)], 32, 128) == 16384 * (1001 + 1002 + 1003)


def test_write_bytes_per_token():
    assert bench.write_bytes(1, 8, 128, 2) == 8192
