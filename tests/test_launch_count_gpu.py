"""The library's own count of the kernels it launches (``fa_launch_count``).

The benchmark reports the kernels launched inside its timed region from this
counter, so the counter must see every launch of every path: one forward
kernel; the backward's row-dot pass, gradient kernel and dQ conversion; a
decoding step's split kernel, plus the combine kernel only when some
(sequence, K/V head) has more than one split.
"""
import pytest
import torch

from exact_attention_21_gb300.inputs import make_qkv
from tests.gpu_util import fa_module

pytestmark = pytest.mark.gpu


def _delta(fa, fn):
    torch.cuda.synchronize()
    before = fa.fa_launch_count()
    out = fn()
    fa.fa_stream_status()
    return fa.fa_launch_count() - before, out


def test_forward_and_backward_launches(cuda_device):
    fa = fa_module()
    t = make_qkv(300, 4, 2, 64, seed=3, with_do=True)
    q, k, v, do = (t[n].to(cuda_device) for n in ("q", "k", "v", "do"))
    n, (o, lse) = _delta(fa, lambda: fa.attention_forward(q, k, v, True))
    assert n == 1
    n, _ = _delta(fa, lambda: fa.attention_backward(q, k, v, o, lse, do, True))
    assert n == 3


@pytest.mark.parametrize("lengths,d,expected", [
    ([200] * 64, 128, 1),   # one split per (sequence, K/V head): the split kernel writes O itself
    ([200] * 64, 64, 1),    # the same on K/V head pairs
    ([20000], 128, 2),      # one long cache: several splits, then the combine
])
def test_decode_launches(cuda_device, lengths, d, expected):
    fa = fa_module()
    B, Hq, Hkv = len(lengths), 64, 8
    N = max(lengths)
    g = torch.Generator().manual_seed(7)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).to(cuda_device)
    k = torch.randn(B * N, Hkv, d, generator=g).to(torch.bfloat16).to(cuda_device)
    v = torch.randn(B * N, Hkv, d, generator=g).to(torch.bfloat16).to(cuda_device)
    n, _ = _delta(fa, lambda: fa.attention_decode(q, k, v, max_seqlen_k=N))
    assert n == expected


def test_failed_call_launches_nothing(cuda_device):
    fa = fa_module()
    q = torch.zeros(16, 2, 64, dtype=torch.bfloat16, device=cuda_device)
    before = fa.fa_launch_count()
    with pytest.raises(fa.FAError):
        # d = 96 is not a supported head dimension: rejected before any launch
        fa.fa_fwd(q, q, q, q, q, 1, 2, 2, 16, 96, 16, 0.1, False, None)
    assert fa.fa_launch_count() == before
