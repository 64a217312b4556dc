"""Host logic of bench.py that needs no GPU: the source hash that ties a
recorded DRAM-traffic figure to the kernel code it was measured on, and the
second staging of a step's inputs for the double-buffered end-to-end loop."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_drops_comments_and_blank_lines_only():
    src = 'int a = 1;  // one\n\n/* two\n   lines */ int b = 2;\nconst char *s = "x // y /* z */";\n'
    assert bench.strip_comments(src) == 'int a = 1;\n  int b = 2;\nconst char *s = "x // y /* z */";'


def test_strip_comments_keeps_character_and_escaped_literals():
    src = "char c = '/'; char d = '*'; const char *e = \"a\\\"//b\"; // gone\n"
    assert bench.strip_comments(src) == "char c = '/'; char d = '*'; const char *e = \"a\\\"//b\";"


def test_comment_edit_keeps_the_hash_and_a_code_edit_changes_it():
    base = "__global__ void k(int *p)\n{\n    p[0] = 1;  // store\n}\n"
    comment_edit = "// a kernel\n__global__ void k(int *p)\n{\n    p[0] = 1;  /* the store */\n}\n"
    code_edit = "__global__ void k(int *p)\n{\n    p[0] = 2;  // store\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(comment_edit)
    assert bench.strip_comments(base) != bench.strip_comments(code_edit)


def test_traffic_is_withheld_for_unrecorded_or_changed_code(monkeypatch):
    assert bench.profiled_traffic("no_such_workload", "paged_decode_kernel") is None
    rec = dict(bench.PROFILED_TRAFFIC)
    key = ("decode_b256", "paged_decode_kernel")
    rec[key] = {"sources_sha256": "0" * 64, "bytes": 1}
    monkeypatch.setattr(bench, "PROFILED_TRAFFIC", rec)
    assert bench.profiled_traffic(*key) is None
    rec[key] = {"sources_sha256": bench.kernel_sources_sha("paged_decode_kernel"), "bytes": 7}
    assert bench.profiled_traffic(*key) == 7


class _FakeStep:
    """The attributes bench.second_stage touches: staged inputs, the output and
    the per-layer tuples (pool, pool, q, k_new, v_new, out)."""


def _staged_step(torch, layers):
    d_all = torch.zeros(4096, dtype=torch.uint8)
    step = _FakeStep()
    step.q = d_all[0:512].view(torch.float16)
    step.lens = d_all[512:640].view(torch.int32)
    step.pool = torch.zeros(64, dtype=torch.float16)  # not staged: shared by both sets
    step.layer_io = []
    if layers:
        outs = [torch.zeros(8, dtype=torch.float16) for _ in range(2)]
        step.layer_io = [(step.pool, step.pool, step.q, step.q, step.q, o) for o in outs]
        step.out = outs[-1]
    else:
        step.out = torch.zeros(8, dtype=torch.float16)
    return d_all, step


def test_second_stage_twins_every_staged_input_and_the_output():
    torch = __import__("torch")
    d_all, step = _staged_step(torch, layers=False)
    q0, lens0, pool0, out0 = step.q, step.lens, step.pool, step.out
    d_all2, use, outs = bench.second_stage(step, d_all, torch)
    assert outs[0] is out0 and outs[1] is not out0 and outs[1].shape == out0.shape
    use(1)
    # the same offsets in the second buffer, not views of the first
    assert step.q.data_ptr() - d_all2.data_ptr() == q0.data_ptr() - d_all.data_ptr()
    assert step.lens.data_ptr() - d_all2.data_ptr() == lens0.data_ptr() - d_all.data_ptr()
    assert step.q.dtype == q0.dtype and step.q.shape == q0.shape
    assert step.pool is pool0 and step.out is outs[1]
    use(0)
    assert step.q is q0 and step.lens is lens0 and step.out is out0


def test_second_stage_gives_each_layer_its_own_output_twin():
    torch = __import__("torch")
    d_all, step = _staged_step(torch, layers=True)
    io0 = list(step.layer_io)
    d_all2, use, outs = bench.second_stage(step, d_all, torch)
    use(1)
    for a, b in zip(io0, step.layer_io):
        assert b[0] is a[0] and b[1] is a[1]        # pools shared
        assert b[2].data_ptr() != a[2].data_ptr()   # q staged twice
        assert b[-1] is not a[-1]                   # each layer's output twinned
    assert outs[1] is step.layer_io[-1][-1]         # the read-back is the last layer's
    use(0)
    assert step.layer_io == io0


def test_prepared_calls_follow_the_buffer_set():
    """The bench's steps are prepared calls cached per buffer set: the second
    staging gets calls prepared on its own buffers, and switching back reuses
    the first set's calls."""
    torch = __import__("torch")
    d_all, step = _staged_step(torch, layers=False)
    step.stage, step.calls = 0, {}
    made = []

    def make():
        made.append((step.q.data_ptr(), step.out))
        return len(made)
    first = bench.Step.prepared(step, ("decode", 0), make)
    assert bench.Step.prepared(step, ("decode", 0), make) == first and len(made) == 1
    d_all2, use, outs = bench.second_stage(step, d_all, torch)
    use(1)
    second = bench.Step.prepared(step, ("decode", 0), make)
    assert second != first and made[1] == (step.q.data_ptr(), outs[1])
    assert made[1][0] != made[0][0]
    use(0)
    assert bench.Step.prepared(step, ("decode", 0), make) == first and len(made) == 2
