"""GPU parity of the bulk-copy ring row pass against the oracle.

Greedy and tree batches of 16-byte-aligned rows larger than 128 MiB stream
through the ring (a producer warp's bulk copies into shared memory); smaller
or unaligned batches take the register path.  These cases put the ring
through fp32 rows, a vocabulary whose last tile is ragged, rows whose pieces
span CTAs, and a large tree; an element-offset copy of the same rows takes the
register path, and both must give the oracle's bit-exact result.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import verify as ov
from tests.gpu_parity import to_device, tokens_to_device

pytestmark = pytest.mark.gpu

RING_MIN_BYTES = 128 * 1024 * 1024


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import speculative_decoding_draft_online_gb300 as sv
    return sv


def greedy_inputs(B, k, V, dtype, seed, a=0.8):
    """Target rows ~ N(0, 4^2) with a planted unique maximum; draft i is row i's
    argmax with probability a, else another id."""
    rng = np.random.default_rng(seed)
    t, top = wl._planted_rows(rng, (B, k + 1), 4.0, V)
    hit = rng.random(size=(B, k)) < a
    tokens = np.where(hit, top[:, :k], wl._other_id(rng, top[:, :k], V)).astype(np.int32)
    return wl.store(t, dtype), tokens


def offset_copy(x: torch.Tensor) -> torch.Tensor:
    """The same values one element past a 16-byte boundary (register path)."""
    flat = torch.empty(x.numel() + 1, dtype=x.dtype, device=x.device)
    y = flat[1:].view(x.shape)
    y.copy_(x)
    return y


def check_greedy(sv, target, tokens, dtype):
    t = to_device(target, dtype)
    x = tokens_to_device(tokens)
    ref = ov.verify_greedy(target, tokens, dtype)
    ok = ref.status == 0
    for dev in (t, offset_copy(t)):
        out, n, aux = sv.verify_ex(dev, None, x, 0.0, 0, aux=True)
        torch.cuda.synchronize()
        out, n = out.cpu().numpy(), n.cpu().numpy()
        np.testing.assert_array_equal(aux["status"].cpu().numpy(), ref.status)
        np.testing.assert_array_equal(out[ok], ref.out_tokens[ok])
        np.testing.assert_array_equal(n[ok], ref.n_accepted[ok])
        assert np.all(n[~ok] == -1) and np.all(out[~ok] == -1)


@pytest.mark.parametrize("dtype,B,k,V", [
    (wl.FP32, 64, 8, 128256),     # fp32 rows: 4096-id tiles of 16 KB, one per stage
    (wl.BF16, 40, 8, 200008),     # ragged last tile; pieces cross row ends
])
def test_ring_greedy_matches_oracle(sv, dtype, B, k, V):
    assert B * (k + 1) * V * (4 if dtype == wl.FP32 else 2) >= RING_MIN_BYTES
    target, tokens = greedy_inputs(B, k, V, dtype, seed=11 + B)
    check_greedy(sv, target, tokens, dtype)


def test_ring_greedy_ties_and_nan(sv):
    """Lowest index among equal maxima, and a NaN row, on the ring path."""
    B, k, V = 64, 8, 128256
    target, tokens = greedy_inputs(B, k, V, wl.BF16, seed=5)
    t = wl.logits_as_f32(target, wl.BF16).reshape(B, k + 1, V).copy()
    t[3, 2, :] = 1.0                        # every id ties
    t[7, 0, 5000] = t[7, 0, 70000] = 50.0   # two equal maxima in different tiles
    t[9, 4, 12345] = np.nan
    tokens[3, 2] = 0
    tokens[7, 0] = 5000
    target = wl.store(t, wl.BF16)
    assert ov.verify_greedy(target, tokens, wl.BF16).status[9] != 0
    check_greedy(sv, target, tokens, wl.BF16)


def test_ring_tree_matches_oracle(sv):
    """The C5 tree shape on 64 sequences (525 MB of rows)."""
    w = wl.c5(seed=205, B=64)
    assert w.target.nbytes >= RING_MIN_BYTES
    ref = ov.verify_tree(w.target, w.tokens, w.parents, w.dtype)
    t = to_device(w.target, w.dtype)
    for dev in (t, offset_copy(t)):
        out, n, leaf, status = sv.verify_tree(dev, tokens_to_device(w.tokens), tokens_to_device(w.parents))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(status.cpu().numpy(), ref.status)
        np.testing.assert_array_equal(out.cpu().numpy(), ref.out_tokens)
        np.testing.assert_array_equal(n.cpu().numpy(), ref.n_accepted)
        np.testing.assert_array_equal(leaf.cpu().numpy(), ref.leaf)
