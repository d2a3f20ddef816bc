"""Pack / unpack on the GPU: bit-exact against a brute-force index map."""
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


def brute_map(lengths):
    order = sorted(range(len(lengths)), key=lambda b: (-lengths[b], b))
    start = np.concatenate([[0], np.cumsum(lengths)])
    src = []
    for t in range(max(lengths)):
        for b in order:
            if lengths[b] > t:
                src.append(start[b] + t)
    return np.array(src, dtype=np.int64)


@pytest.mark.parametrize("lengths", [[3, 1, 4, 0, 2], [1], [0, 5, 0], list(range(1, 130)),
                                     list(np.random.default_rng(3).integers(0, 300, 257))])
@pytest.mark.parametrize("dtype,width", [(torch.float32, 4), (torch.float32, 40), (torch.bfloat16, 8),
                                         (torch.bfloat16, 64)])
def test_pack_is_the_index_map_and_unpack_inverts_it(lengths, dtype, width):
    from padding_free_variable_gb300 import ops
    lengths = [int(v) for v in lengths]
    plan = ops.Plan(lengths)
    N = sum(lengths)
    x = torch.randn(N, width, device="cuda").to(dtype)
    xp = plan.pack(x)
    src = brute_map(lengths)
    assert xp.shape[0] == len(src)
    assert torch.equal(xp.cpu(), x.cpu()[torch.from_numpy(src)])
    back = plan.unpack(xp)
    assert torch.equal(back.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       x.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))


def test_arange_packs_to_offsets():
    """Packing the frame index itself yields exactly off[t]+j <-> cstart[perm[j]]+t."""
    from padding_free_variable_gb300 import ops
    lengths = [4, 7, 1, 7, 3]
    plan = ops.Plan(lengths)
    N = sum(lengths)
    x = torch.arange(N, dtype=torch.float32, device="cuda").repeat(4, 1).t().contiguous()
    xp = plan.pack(x)[:, 0].cpu().numpy().astype(int)
    bs, off, perm, slot_len = plan.tables()
    cstart = np.concatenate([[0], np.cumsum(lengths)])
    for t in range(plan.steps):
        for j in range(bs[t]):
            assert xp[off[t] + j] == cstart[perm[j]] + t


def test_padded_pack_zero_fills():
    from padding_free_variable_gb300 import ops
    lengths = [2, 0, 3]
    plan = ops.Plan(lengths, padded=True)
    x = torch.arange(1, 6, dtype=torch.float32, device="cuda").repeat(4, 1).t().contiguous()
    xp = plan.pack(x)[:, 0].cpu().numpy()
    assert list(xp) == [1, 0, 3, 2, 0, 4, 0, 0, 5]
    back = plan.unpack(plan.pack(x))
    assert torch.equal(back, x)
