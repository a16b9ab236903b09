"""Host logic of bench.py that needs no GPU: the validity rule of the
recorded DRAM traffic (keyed to the decode kernel's code, not its comments)
and the per-step category ledger."""
import json
import shutil
from pathlib import Path

import pytest

import bench


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and the traffic record under a scratch
    root, with bench pointed at it."""
    src = tmp_path / "mla_decode_attention_run_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in bench.DECODE_SOURCES:
        shutil.copy(f"{bench.ROOT}/mla_decode_attention_run_gb300/csrc/{name}", src / name)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # a record taken on exactly these sources
    with open(f"{Path(__file__).resolve().parent.parent}/profiles/decode_traffic.json") as f:
        d = json.load(f)
    d["kernel_source_sha"] = bench.decode_source_hash()
    with open(tmp_path / "profiles" / "decode_traffic.json", "w") as f:
        json.dump(d, f)
    return tmp_path


def _record(root):
    with open(root / "profiles" / "decode_traffic.json") as f:
        return json.load(f)


def test_committed_record_is_used_only_on_its_kernel():
    d = _record(Path(bench.ROOT))
    assert d["dram_bytes_per_launch"] == d["dram_read_bytes"] + d["dram_write_bytes"]
    got = bench.committed_traffic(d["workload"])
    if d["kernel_source_sha"] == bench.decode_source_hash():
        assert got == d["dram_bytes_per_launch"]
    else:                                           # taken on other code: not reported
        assert got is None


def test_comment_edits_keep_the_record(tree):
    d = _record(tree)
    f = tree / "mla_decode_attention_run_gb300" / "csrc" / "decode_tc.cu"
    text = f.read_text()
    assert "constexpr int kStages = 4;\n" in text
    text = text.replace("constexpr int kStages = 4;\n", "constexpr int kStages = 4;   // a trailing note\n\n")
    f.write_text("// a new leading comment\n\n" + text + "\n/* a block\n   comment */\n")
    assert bench.decode_source_hash() == d["kernel_source_sha"]
    assert bench.committed_traffic(d["workload"]) == d["dram_bytes_per_launch"]


def test_code_edits_void_the_record(tree):
    d = _record(tree)
    f = tree / "mla_decode_attention_run_gb300" / "csrc" / "decode_params.h"
    f.write_text(f.read_text().replace("int32_t n_blocks;", "int32_t n_blocks, n_extra;"))
    assert bench.decode_source_hash() != d["kernel_source_sha"]
    assert bench.committed_traffic(d["workload"]) is None


def test_another_workload_gets_no_traffic(tree):
    assert bench.committed_traffic("decode_step_b1_h16_l78") is None


def test_category_ledger():
    led = bench.category_ledger(10.0, {"store": 0.5, "attention": 8.0})
    assert led["step_ms"] == 10.0
    assert led["categories"]["attention"] == {"ms": 8.0, "share": 0.8, "step_ms_if_free": 2.0}
    assert led["categories"]["store"]["share"] == 0.05
    assert led["other_ms"] == 1.5
    # a category can't free more than the whole step
    assert bench.category_ledger(1.0, {"cast": 1.2})["categories"]["cast"]["step_ms_if_free"] == 0.0
