"""Replays the golden allocator scripts (tests/golden/*.json) against any
block manager exposing add / fork / free / alloc_slots / block_table / filled /
ref / free-queue views.  Shared by the oracle tests and the C-ABI tests; it
holds no allocator logic, only the expected values from the pages."""
import json
import os


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def replay(doc, mgr):
    """``mgr`` is an adapter with methods add, fork, free, alloc_slots,
    table(seq), filled(seq), ref(block), free_queue()."""
    for step in doc["ops"]:
        op = step["op"]
        if op == "add":
            slots = mgr.add(step["seq"], step["n"])
            if "expect_slots" in step:
                assert list(slots) == step["expect_slots"], step
            if "expect_table" in step:
                assert mgr.table(step["seq"]) == step["expect_table"], step
            if "expect_filled" in step:
                assert mgr.filled(step["seq"]) == step["expect_filled"], step
        elif op == "fork":
            mgr.fork(step["parent"], step["child"])
        elif op == "free":
            mgr.free(step["seq"])
        elif op == "alloc_slots":
            slots, copies = mgr.alloc_slots(step["seqs"])
            assert list(slots) == step["expect_slots"], step
            assert [list(c) for c in copies] == step["expect_copies"], step
        else:
            raise AssertionError(op)
        for s, t in step.get("expect_table", {}).items() if isinstance(step.get("expect_table"), dict) else []:
            assert mgr.table(int(s)) == t, (step, s)
        for s, f in step.get("expect_filled", {}).items() if isinstance(step.get("expect_filled"), dict) else []:
            assert mgr.filled(int(s)) == f, (step, s)
        for b, r in step.get("expect_ref", {}).items():
            assert mgr.ref(int(b)) == r, (step, b)
        if "expect_blocks_in_use" in step:
            n = doc["num_blocks"] - len(mgr.free_queue())
            assert n == step["expect_blocks_in_use"], step
        if "expect_free_tail" in step:
            tail = step["expect_free_tail"]
            assert mgr.free_queue()[-len(tail):] == tail, (step, mgr.free_queue())
