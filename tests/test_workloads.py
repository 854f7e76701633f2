"""Host-side checks of the seeded workload table (no GPU, no oracle)."""
import torch

from causal_prefill_flash_gb300 import workloads as W


def test_table_shapes_and_counts():
    names = [w.name for w in W.WORKLOADS]
    assert len(names) == len(set(names)) == 9
    c = {w.name: w for w in W.WORKLOADS}
    # algorithmic FLOPs = 4 * hd * visible (row, key) pairs
    assert c["single_head_s256"].flops() == 4 * 128 * (256 * 257 // 2)
    assert c["prefill7b_s2048"].flops() == 4 * 128 * 32 * (2048 * 2049 // 2)
    assert c["ragged_s2659_std3"].flops() == 4 * 128 * 32 * (2659 * 2660 // 2)
    assert c["gqa_s8192_bf16"].flops() == 4 * 128 * 32 * (8192 * 8193 // 2)
    # chunked: row i sees 7680 + i + 1 keys
    per_head = sum(7681 + i for i in range(512))
    assert c["chunked_kv8192_hd128"].flops() == 4 * 128 * 4 * 32 * per_head
    assert c["chunked_kv8192_hd64"].flops() == 4 * 64 * 4 * 32 * per_head
    # long context: row i of the 128-row chunk sees 32640 + i + 1 keys
    assert c["longctx_chunk128_kv32768"].flops() == 4 * 128 * 32 * sum(32641 + i for i in range(128))
    # no mask: every row sees every key
    assert c["encoder_s4096_noncausal"].flops() == 4 * 128 * 2 * 16 * 4096 * 4096
    assert c["gqa_s4096_hd256_bf16"].flops() == 4 * 256 * 16 * (4096 * 4097 // 2)


def test_inputs_are_seeded_and_typed():
    w = W.get("single_head_s256")
    q1, k1, v1 = W.make_inputs(w)
    q2, k2, v2 = W.make_inputs(w)
    assert q1.dtype == torch.float16 and q1.shape == (1, 256, 1, 128)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.equal(q1, k1)
    small = W.WORKLOADS[3].with_(Sq=16, Skv=16)
    q, k, v = W.make_inputs(small)
    assert q.dtype == torch.bfloat16 and k.shape == (1, 16, 8, 128)
    rag = W.get("ragged_s2659_std3").with_(Sq=300, Skv=300, Hq=2, Hkv=2)
    q, k, v = W.make_inputs(rag)
    assert 2.5 < q.float().std().item() < 3.5 and 0.8 < v.float().std().item() < 1.2


def test_sample_rows_cover_corners():
    w = W.get("gqa_s8192_bf16")
    rows = W.sample_rows(w, 64)
    assert rows.shape == (64, 3)
    s = {tuple(r.tolist()) for r in rows}
    assert (0, 0, 0) in s and (0, 31, 8191) in s
    assert int(rows[:, 2].max()) < w.Sq and int(rows[:, 1].max()) < w.Hq
