"""A multi-layer decode step: several attention layers, each with its own pool,
q and new K/V, sharing the sequences' block tables, lengths and slots (the
Qwen2.5-0.5B stack has 24).  Each layer must match the oracle; replaying the
whole stack from one CUDA graph must give the same bits as running it eagerly."""
import numpy as np
import pytest
import torch

import _gpu
from _gpu import DevStep, compare
from paged_kv_decode_ns_gb300 import binding as nb
from paged_kv_decode_ns_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_layer_stack_matches_oracle_and_graph_replay(orc):
    st = wl.WORKLOADS["decode_b32"]()
    layers = wl.layer_steps(st, 3)
    devs = [DevStep(layer) for layer in layers]
    for d in devs[1:]:  # one copy of the per-sequence tensors, as in a model
        d.block_tables, d.context_lens, d.slot_mapping = (devs[0].block_tables, devs[0].context_lens,
                                                          devs[0].slot_mapping)
    ws = devs[0].ws  # one workspace serves the whole stack

    def step():
        for d in devs:
            nb.ns_kv_append_paged_attn_decode(d.q, d.k_new, d.v_new, d.slot_mapping, d.k_pool,
                                              d.v_pool, d.block_tables, d.context_lens, d.st.scale,
                                              d.out, ws)

    step()
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    eager = [d.out.clone() for d in devs]
    for layer, d in zip(layers, devs):
        ref, kp, vp = orc.step(layer, num_threads=max(1, orc.max_threads()))
        compare(d.out, ref, layer.dtype, layer.name)
        assert np.array_equal(_gpu.to_bits(d.k_pool), kp), layer.name
        assert np.array_equal(_gpu.to_bits(d.v_pool), vp), layer.name

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm the capture stream's path
    torch.cuda.synchronize()
    for d in devs:
        d.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    for layer, e, d in zip(layers, eager, devs):
        assert torch.equal(e.view(torch.int16), d.out.view(torch.int16)), layer.name
    _gpu.assert_no_device_status()


def test_layer_stack_with_overlapped_prologues_gives_the_same_bits(orc):
    """Launched as programmatic dependents (each layer's prologue may overlap the
    previous layer's tail), eagerly and from a CUDA graph, the stack gives the
    bits of plain launches."""
    st = wl.WORKLOADS["decode_b32"]()
    layers = wl.layer_steps(st, 4)
    plain = [DevStep(layer) for layer in layers]
    over = [DevStep(layer) for layer in layers]
    cfg = nb.DecodeConfig()
    cfg.overlap_prologue = 1

    def run(devs, config):
        for d in devs:
            nb.ns_kv_append_paged_attn_decode(d.q, d.k_new, d.v_new, d.slot_mapping, d.k_pool,
                                              d.v_pool, d.block_tables, d.context_lens, d.st.scale,
                                              d.out, devs[0].ws, config=config)

    run(plain, None)
    run(over, cfg)
    torch.cuda.synchronize()
    _gpu.assert_no_device_status()
    for layer, a, b in zip(layers, plain, over):
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16)), layer.name
        assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16)), layer.name
    ref, _, _ = orc.step(layers[2], num_threads=max(1, orc.max_threads()))
    compare(over[2].out, ref, layers[2].dtype, layers[2].name)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(over, cfg)
    torch.cuda.synchronize()
    for d in over:
        d.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(over, cfg)
    g.replay()
    torch.cuda.synchronize()
    for layer, a, b in zip(layers, plain, over):
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16)), layer.name
    _gpu.assert_no_device_status()
