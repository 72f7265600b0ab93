"""The schedule tool (no GPU): the canonical artifact is deterministic, round
trips through JSON without changing the validator's decision, and identifies
a schedule by its hash."""
import json

import pytest


@pytest.fixture(scope="module")
def tool():
    from decode_megakernel_02_gb300 import build
    build.build()
    from decode_megakernel_02_gb300 import schedule
    schedule.mk.load()
    return schedule


def test_artifact_is_deterministic(tool):
    a, b = tool.lower("tiny", 7, 3), tool.lower("tiny", 7, 3)
    assert tool.canonical(a) == tool.canonical(b)
    assert tool.digest(a) == tool.digest(b)
    assert tool.digest(tool.lower("tiny", 7, 2)) != tool.digest(a)
    assert tool.digest(tool.lower("tiny", 8, 3)) != tool.digest(a)


def test_round_trip_keeps_the_schedule(tool):
    ir = tool.lower("tiny", 152, 0)
    back = tool.from_canonical(tool.canonical(ir))
    assert tool.digest(back) == tool.digest(ir)
    assert tool.mk.mk_validate_ir(back)[0] == tool.mk.MK_OK
    assert back["tagged"] == ir["tagged"] and back["tagged"]


def test_dumped_schedule_is_validated_again(tool, tmp_path):
    out = tmp_path / "ir.json"
    assert tool.main(["dump", "--workload", "tiny", "--sms", "7", "--chunks", "3", "--out", str(out)]) == 0
    assert tool.main(["validate", "--ir", str(out)]) == 0
    doc = json.loads(out.read_text())
    t = next(t for t in doc["tasks"] if t["waits"])
    t["waits"][0][1] += 1  # one more signal than the counter has producers
    out.write_text(json.dumps(doc))
    assert tool.main(["validate", "--ir", str(out)]) == 1


def test_explain_counts(tool):
    ir = tool.lower("llama-1b", 152, 0)
    e = tool.explain(ir)
    assert e["decoder_layers"] == 16 and e["ctas"] == 152 and e["tasks"] == len(ir["tasks"])
    assert e["tasks_per_op"]["attn"] == 16 * 8 * 6  # layers x KV heads x chunks
    assert e["tagged_counters"] == 16
    assert sum(e["tasks_per_op"].values()) == e["tasks"]
