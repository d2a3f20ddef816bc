"""The tcgen05 input projection (bf16 operands, fp32 accumulation in tensor
memory) against an fp64 product of the same bf16 values, and against the
CUDA-core engine, on ragged shapes (M not a multiple of 128, N not a multiple
of 256, K below and above one 64-wide k-block and not a multiple of it).

Bar: fp32 accumulation of K exact bf16 products differs from the fp64 sum by
at most about K * 2^-24 of the sum of |terms|; 1e-5 of the output's scale
covers K <= 2048 here.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


SHAPES = [  # rows M, input D (=K), hidden H, directions (N = nd*4H)
    (1000, 40, 512, 2),
    (129, 64, 80, 1),
    (4096, 1024, 256, 2),
    (777, 72, 136, 2),
    (18149, 2048, 64, 2),
]


@pytest.mark.parametrize("M,D,H,nd", SHAPES)
def test_tensor_core_projection_matches_fp64(M, D, H, nd):
    from padding_free_variable_gb300 import ops, synthetic
    from gpu_harness import rel_err
    rng = np.random.default_rng(M + D + H)
    x = synthetic.round_bf16(rng.standard_normal((M, D)).astype(np.float32))
    W = synthetic.round_bf16(rng.uniform(-0.1, 0.1, (nd, 4 * H, D)).astype(np.float32))
    b = rng.uniform(-0.1, 0.1, (nd, 4 * H)).astype(np.float32)
    plan = ops.Plan([M])
    shape = ops.layer_shape(D, H, nd, True)
    layer = {"W": torch.from_numpy(W).to("cuda", torch.bfloat16), "R": torch.zeros((nd, 4 * H, H), device="cuda",
             dtype=torch.bfloat16), "b": torch.from_numpy(b).cuda(), "peep": torch.zeros((nd, 3, H), device="cuda")}
    xd = torch.from_numpy(x).to("cuda", torch.bfloat16)
    outs = {}
    for engine in (0, 1):
        plan.set_gemm_engine(engine)
        out = torch.full((M, nd * 4 * H), float("nan"), device="cuda")
        ops.input_projection(plan, shape, layer, xd, out)
        torch.cuda.synchronize()
        assert plan.poll() == 0
        outs[engine] = out.cpu().numpy()
    ref = x.astype(np.float64) @ W.reshape(nd * 4 * H, D).astype(np.float64).T + b.reshape(-1)
    assert np.all(np.isfinite(outs[0]))
    assert rel_err(outs[0], ref) <= 1e-5
    assert rel_err(outs[1], ref) <= 1e-5
    assert rel_err(outs[0], outs[1]) <= 1e-5
