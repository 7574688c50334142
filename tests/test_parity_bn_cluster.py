"""BatchNorm2d through the cluster kernels (a thread-block cluster of K = 2,
4 or 8 blocks per channel, partial sums exchanged in distributed shared
memory) against the float64 oracle.

The composite calls take these kernels for channels of more than
bn_small_max_elems() and at most 8 x that many elements, while the C*K
blocks fit one per SM (below the persistent kernel's threshold);
lowering the limit forces every cluster size on small shapes.  Shapes are ragged (channel sizes that no cluster size
divides evenly) in fp32 and bf16, with and without a fused activation; the
largest eligible channel and the first one past it (which takes the
two-launch kernels) are checked too, and a second run must give the same
bits."""

import pytest
import torch

from bwd_bn_pass_gb300 import synth

from . import test_parity_bn as base
from . import test_parity_bn_act as act_base

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture
def limit(gbn):
    """Sets the per-block element limit for one test (the persistent kernel
    out of reach), restoring both settings afterwards."""
    prev_p = gbn.bn_set_persistent_min_bytes(1 << 62)
    prev_s = gbn.bn_small_max_elems()

    def set_limit(m):
        gbn.bn_set_small_max_elems(m)
        return gbn.bn_small_max_elems()

    yield set_limit
    gbn.bn_set_small_max_elems(prev_s)
    gbn.bn_set_persistent_min_bytes(prev_p)


# (B, C, H, W): M = B*H*W = 2015 (fp32) and 1938 (bf16); limits giving
# clusters of 1 (the one-block kernel), 2, 4 and 8 blocks per channel
SHAPES = {"f32": (5, 7, 13, 31), "bf16": (6, 10, 17, 19)}
LIMITS = [2048, 1008, 504, 252]


def _blocks(M, lim):
    for K in (1, 2, 4, 8):
        if -(-M // K) <= lim:
            return K
    return 0


@pytest.mark.parametrize("lim", LIMITS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cluster_parity_every_cluster_size(gbn, limit, dtype, lim):
    shape = SHAPES[dtype]
    M = shape[0] * shape[2] * shape[3]
    assert limit(lim) == lim
    K = [1, 2, 4, 8][LIMITS.index(lim)]
    assert _blocks(M, lim) == K
    assert gbn.bn_small_blocks_per_channel(shape) == K
    case = synth.BNCase(f"cluster_{dtype}_{lim}", shape, dtype, mu_range=(-50.0, 50.0),
                        sigma_range=(0.01, 5.0), seed=5100 + lim)
    inp = synth.bn_inputs(case)
    got = base.run_gpu(gbn, inp)
    base.compare(got, base.run_oracle(inp), dtype, what=f"{case.name}")
    again = base.run_gpu(gbn, inp)
    for k in got:
        assert torch.equal(got[k], again[k]), f"{case.name} {k} differs between runs"


def test_cluster_size_choice():
    """The cluster sizes the shapes above exercise (host arithmetic only)."""
    for dtype, shape in SHAPES.items():
        M = shape[0] * shape[2] * shape[3]
        assert [_blocks(M, lim) for lim in LIMITS] == [1, 2, 4, 8], dtype


@pytest.mark.parametrize("lim", [1008, 252])
@pytest.mark.parametrize("act", ["relu", "leaky_relu"])
def test_cluster_act_parity(gbn, limit, act, lim):
    limit(lim)
    case = synth.BNCase(f"cluster_act_{lim}", SHAPES["f32"], "f32", mu_range=(-5.0, 5.0),
                        sigma_range=(0.1, 3.0), seed=5200 + lim)
    inp = synth.bn_inputs(case)
    act_base.nudge_off_kink(inp)
    slope = act_base.ACTS[act][1]
    act_base.compare(act_base.run_gpu(gbn, inp, act, slope),
                     act_base.run_oracle(inp, act, slope), "f32", what=f"{case.name} {act}")


@pytest.mark.parametrize("shape", [(16, 3, 32, 32), (16, 3, 32, 32 + 1)],
                         ids=["M=16384 (8 blocks of 2048)", "M=16896 (two-launch)"])
def test_cluster_largest_channel_and_past_it(gbn, limit, shape):
    limit(2048)
    assert gbn.bn_small_blocks_per_channel(shape) == (8 if shape[3] == 32 else 0)
    case = synth.BNCase("cluster_edge", shape, "f32", mu_range=(-1e3, 1e3),
                        sigma_range=(0.01, 10.0), seed=5300 + shape[3])
    inp = synth.bn_inputs(case)
    base.compare(base.run_gpu(gbn, inp), base.run_oracle(inp), "f32", what=str(shape))


def test_cluster_ragged_default(gbn, limit):
    """[3,37,41,40] (4920 elements per channel) at the default limit: a
    cluster of four blocks per channel."""
    assert limit(2048) == 2048
    assert gbn.bn_small_blocks_per_channel((3, 37, 41, 40)) == 4
    case = synth.CASES["bn_ragged_f32"]
    inp = synth.bn_inputs(case)
    base.compare(base.run_gpu(gbn, inp), base.run_oracle(inp), "f32", what="ragged")


def test_one_wave_rule(gbn, limit):
    """The small-channel kernels take a shape only while its blocks form a
    single wave: one block per channel up to 4 blocks per SM, clusters up to
    one block per SM; past that the two-launch kernels run, with the same
    results."""
    limit(2048)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cmax1 = 4 * sms       # one block per channel (M <= 2048)
    cmax4 = sms // 4      # clusters of four (4096 < M <= 8192)
    assert gbn.bn_small_blocks_per_channel((2, cmax1, 32, 32)) == 1
    assert gbn.bn_small_blocks_per_channel((2, cmax1 + 1, 32, 32)) == 0
    assert gbn.bn_small_blocks_per_channel((8, cmax4, 32, 32)) == 4
    assert gbn.bn_small_blocks_per_channel((8, cmax4 + 1, 32, 32)) == 0
    for shape in ((2, cmax1 + 1, 8, 8), (8, cmax4 + 1, 32, 32)):
        case = synth.BNCase("one_wave", shape, "f32", mu_range=(-10.0, 10.0),
                            sigma_range=(0.1, 2.0), seed=5400 + shape[1])
        inp = synth.bn_inputs(case)
        base.compare(base.run_gpu(gbn, inp), base.run_oracle(inp), "f32", what=str(shape))
