"""A decode through a stack of layers in one CUDA graph, each layer's output the next layer's input.

The page "Qwen3.6-35B-A3B (qwen3_5_moe) on the native Metal engine: proposal and gate" decodes whole stacks
of these layers (slice "The lane host and the prompt cache"), and the model's MTP layer is one more layer of
the same shape.  Here four layers of the decode shape, each with its own weights, are chained through
moe_forward on one stream and one workspace: called one by one, then captured in a CUDA graph and replayed.
Between two layers each output row is scaled to unit RMS (plain PyTorch ops in the same stream and graph, a
stand-in for the model's norm, without which the rows grow quadratically from layer to layer).  The graph's
bytes must equal the call-by-call bytes, and every layer's output must match the oracle run on that layer's
own input as the GPU saw it.  The chain exercises back-to-back launches sharing a workspace (its counters and
launch epoch carry over from one layer to the next).
"""
import numpy as np
import pytest
import torch

import oracle
import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu

LAYERS = 4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    qm.load()
    oracle.build()


@pytest.mark.parametrize("T", [1, 16])
def test_layer_chain_in_one_graph(T):
    shape = synth.QWEN_SHAPE
    weights = [synth.make_weights(shape, 100 + l) for l in range(LAYERS)]
    layers = [qm.DeviceLayer(w) for w in weights]
    x0 = synth.make_x(shape, T, 100, stream=T)
    dev = "cuda"
    xs = [torch.from_numpy(x0.view(np.int16)).to(dev)]
    xs += [torch.empty((T, shape.hidden), dtype=torch.int16, device=dev) for _ in range(LAYERS - 1)]
    ys = [torch.empty((T, shape.hidden), dtype=torch.int16, device=dev) for _ in range(LAYERS)]
    ids = [torch.empty((T, shape.top_k), dtype=torch.int32, device=dev) for _ in range(LAYERS)]
    p = [torch.empty((T, shape.top_k), dtype=torch.int16, device=dev) for _ in range(LAYERS)]
    w_s = [torch.empty((T,), dtype=torch.int16, device=dev) for _ in range(LAYERS)]
    ws = qm.workspace(layers[0].cfg, T)
    stream = torch.cuda.Stream()

    def chain():
        for l in range(LAYERS):
            qm.moe_forward(layers[l].cfg, layers[l].w, xs[l], T, None, None, ys[l], ids[l], p[l], w_s[l],
                           qm.MOE_PATH_AUTO, ws, stream)
            if l + 1 < LAYERS:
                yf = ys[l].view(torch.bfloat16).float()
                xn = yf * torch.rsqrt((yf * yf).mean(dim=1, keepdim=True))
                xs[l + 1].copy_(xn.to(torch.bfloat16).view(torch.int16))

    def outputs():
        return [dict(x=H.u16(xs[l]), y=H.u16(ys[l]), ids=ids[l].cpu().numpy(), p=H.u16(p[l]), w_s=H.u16(w_s[l]))
                for l in range(LAYERS)]

    with torch.cuda.stream(stream):
        chain()
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    solo = outputs()
    for t in xs[1:] + ys + p + w_s:
        t.zero_()
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            chain()
    for _ in range(2):                       # replayed twice: the workspace state carries over between replays
        graph.replay()
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    got = outputs()
    for l in range(LAYERS):
        for key in ("x", "y", "ids", "p", "w_s"):
            assert np.array_equal(got[l][key], solo[l][key]), (l, key)

    # each layer against the oracle on its own input as the GPU saw it
    for l in range(LAYERS):
        _check_layer(shape, weights[l], layers[l], got[l]["x"], got[l])


def _check_layer(shape, w, layer, x_bits, got):
    """ids on unambiguous rows, p and w_s within one bf16 ulp, y by the output rule relative to each row's
    scale; near-tie rows under the GPU's own logits."""
    ref = oracle.forward(shape, w, x_bits)
    clear = H.oracle_gap(ref["logits"], shape.top_k) >= H.AMBIGUOUS_GAP
    assert np.array_equal(got["ids"][clear], ref["ids"][clear])
    same = np.nonzero(np.all(got["ids"] == ref["ids"], axis=1))[0]
    assert H.ulp_diff_bf16(got["p"][same], ref["p"][same]).max(initial=0) <= 1
    assert H.ulp_diff_bf16(got["w_s"], ref["w_s"]).max(initial=0) <= 1
    H.check_rows_scale_free(got["y"][same], ref["y"][same])
    diff = np.nonzero(np.any(got["ids"] != ref["ids"], axis=1))[0]
    if len(diff):
        r = H.run_route(layer, x_bits)
        assert np.array_equal(r["ids"], got["ids"])
        ref2 = oracle.forward(shape, w, x_bits, logits_in=r["logits"], rows=diff)
        assert np.array_equal(ref2["ids"], got["ids"][diff])
        assert np.array_equal(ref2["p"], got["p"][diff])
        H.check_rows_scale_free(got["y"][diff], ref2["y"])
    rms = np.sqrt((H.bf16_to_f64(ref["y"]) ** 2).mean())
    print(f"layer output rms {rms:.3g}, near-tie rows {len(diff)}")
