"""The bench's byte accounting against the Quest page's §2 numbers."""

import bench


def test_paper_ratio_and_bytes(golden):
    ex = golden("byte_model.json")
    assert bench.paper_traffic_ratio(ex["L"], ex["S"], ex["budget_tokens"]) == ex["rho"]
    # one layer, one KV head, 64K tokens, budget 4096: 2 MiB summary + 2 MiB K/V
    b = bench.step_bytes(ex["L"] // ex["S"], 1, 1, 128, ex["S"], ex["K"], ex["K"] * ex["S"], 2)
    assert b["summary"] == ex["index_MiB"] << 20
    assert b["kv"] == ex["selected_MiB"] << 20


def test_llama_layer_step_bytes():
    b = bench.step_bytes(2048, 32, 1, 128, 16, 128, 128 * 16, 2)
    assert b["summary"] == 32 << 20 and b["kv"] == 32 << 20
    assert b["q"] == 8192 and b["o"] == 16384
    assert 67.1e6 < b["total"] < 67.3e6


def test_e4m3_summary_halves_the_index_term():
    """E4M3 codes are one byte per summary element: the index term (eq (10))
    halves against fp16 and nothing else changes."""
    a = bench.step_bytes(2048, 32, 1, 128, 16, 128, 128 * 16, 2)
    b = bench.step_bytes(2048, 32, 1, 128, 16, 128, 128 * 16, 2, summary_esize=1)
    assert b["summary"] * 2 == a["summary"] == 2048 * 32 * 2 * 128 * 2
    assert b["kv"] == a["kv"] and b["q"] == a["q"] and b["o"] == a["o"]
    assert a["append"] - b["append"] == 32 * 2 * 128 * 2
