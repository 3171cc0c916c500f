"""ResNet-50 forward through the C ABI: every layer checked against the
oracle on the GPU's own layer input (so errors do not compound), at sampled
outputs for the large layers; pools and the FC checked in full."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def test_resnet50_layerwise_parity():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.resnet50 import ResNet50
    dev = torch.device("cuda:0")
    N = 2
    net = ResNet50(N, dev, seed=3, algo="auto", keep=True)
    assert len(net.specs) == 54  # 53 convs + the FC
    x = synth.normal((N, 3, 224, 224), 1.0, 5)
    logits = net.forward(torch.from_numpy(x).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    t = {k: v.double().cpu().numpy() for k, v in net.tensors.items()}
    # boundary conversion: NCHW fp32 -> NHWC bf16 with 3 channels padded to 8
    assert np.array_equal(t["input"][..., :3], nchw_to_nhwc(ol.round_bf16(x)))
    assert np.all(t["input"][..., 3:] == 0)
    g = np.random.default_rng(0)
    worst = {}
    for sp in net.specs:
        xin = nhwc_to_nchw(t[sp.src])
        w = nhwc_to_nchw(net.weights[sp.name].double().cpu().numpy())
        b = net.biases[sp.name].double().cpu().numpy()
        res = nhwc_to_nchw(t[sp.residual]) if sp.residual else None
        y = t[sp.dst]
        OH, OW = y.shape[1], y.shape[2]
        P = 512
        idx = np.stack([g.integers(0, N, P), g.integers(0, sp.K, P), g.integers(0, OH, P),
                        g.integers(0, OW, P)], axis=1)
        ref = ol.conv2d_f64_points(xin, w, idx, b, stride=sp.stride, pad=sp.pad,
                                   residual=res, act=1 if sp.act else 0)
        got = y[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
        denom = max(np.max(np.abs(ref)), 1e-30)
        err = np.max(np.abs(got - ref)) / denom
        worst[sp.name] = err
        assert err <= 1e-2, (sp.name, net.algos[sp.name], err)
    # max pool (exact) and global average pool
    mp = nchw_to_nhwc(ol.maxpool2d(nhwc_to_nchw(t["conv1"]), 3, 2, 1))
    assert np.array_equal(t["pool1"], mp)
    ap = ol.global_avgpool(nhwc_to_nchw(t[net.specs[-2].dst]))
    np.testing.assert_allclose(t["pool5"].reshape(N, 2048), ap, rtol=1e-2, atol=1e-2)
    assert logits.shape == (N, 1000) and torch.isfinite(logits.float()).all()


def test_resnet50_cuda_graph_replay_matches_eager():
    """A captured forward replays to the same logits as the eager forward, and
    picks up new input values written into the captured input buffer."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.resnet50 import ResNet50
    dev = torch.device("cuda:0")
    net = ResNet50(2, dev, seed=4, algo="auto")
    x = torch.from_numpy(synth.normal((2, 3, 224, 224), 1.0, 6)).to(dev)
    eager = net.forward(x).clone()
    out = net.capture(x.clone())
    net._graph_x.copy_(x)
    got = net.replay()
    torch.cuda.synchronize()
    assert torch.equal(got, eager)
    x2 = torch.from_numpy(synth.normal((2, 3, 224, 224), 1.0, 7)).to(dev)
    eager2 = net.forward(x2).clone()
    net._graph_x.copy_(x2)
    got2 = net.replay()
    torch.cuda.synchronize()
    assert torch.equal(got2, eager2) and not torch.equal(got2, eager)
    # a second, independent graph over another input buffer (the end-to-end
    # bench alternates two): each replays its own buffer, back to back
    xb = x.clone()
    g2, out2 = net.capture_graph(xb)
    net._graph_x.copy_(x2)
    net.replay()
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, eager) and torch.equal(net._graph_out, eager2)
    del out
