"""Guard bands around every output buffer.

With no memory sanitizer on this GPU, out-of-range stores are caught the
plain way: each output (O, LSE, dQ, dK, dV, the backward workspace, the
decode split buffer) is carved out of a larger allocation whose 4 KiB before
and after it hold a sentinel byte pattern, and after the call those bands
must be bit for bit unchanged.  The cases are the ones where a store could
run past its tensor: ragged tails (N = 1, 127, 129, 200), padded batches
with an empty sequence and a query-less one, unequal query and key lengths,
decode over 1 and 20000 keys, and the FP8, bf16-output, masked and
allocation-free entry points.  ("FlashAttention Interview Questions",
section "Does subtracting the maximum solve every numerical issue?": tile
boundaries, padding and masked positions are where such defects hide.)
"""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import scale_for

pytestmark = pytest.mark.gpu

BAND = 4096          # bytes of sentinel before and after each output
SENTINEL = 0xA5


class Banded:
    """A tensor view inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.buf = torch.full((BAND + nbytes + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.nbytes = nbytes
        self.t = self.buf[BAND:BAND + nbytes].view(dtype).view(shape)

    def bands_intact(self):
        b = self.buf.cpu()
        return bool(torch.all(b[:BAND] == SENTINEL)) and bool(torch.all(b[BAND + self.nbytes:] == SENTINEL))


def _check(what, *banded):
    torch.cuda.synchronize()
    fa.sync_status()
    for i, b in enumerate(banded):
        assert b.bands_intact(), f"{what}: output {i} wrote outside its buffer"


@pytest.mark.parametrize("N", [1, 127, 129, 200])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_backward_ragged(N, d, causal):
    B, H = 1, 2
    inp = workloads.make_inputs(B, H, N, d, seed=400 + N + d, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    o, lse = Banded((B, H, N, d), torch.float32), Banded((B, H, N), torch.float32)
    fa.forward(q, k, v, causal=causal, scale=scale, out=(o.t, lse.t))
    _check(("fwd", N, d, causal), o, lse)
    g = [Banded((B, H, N, d), torch.float32) for _ in range(3)]
    ws = Banded((B * H * N,), torch.float32)
    fa.backward(q, k, v, o.t, lse.t, do, causal=causal, scale=scale, workspace=ws.t, out=tuple(x.t for x in g))
    _check(("bwd", N, d, causal), *g, ws)
    assert all(torch.isfinite(x.t).all() for x in g)


@pytest.mark.parametrize("causal", [False, True])
def test_padded_batch_with_empty_sequences(causal):
    B, H, Nq, Nk, d = 4, 2, 300, 260, 128
    sq, sk = [300, 0, 129, 41], [260, 77, 0, 200]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=411)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    do = workloads.randn_bf16((B, H, Nq, d), 413).cuda()
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    scale = scale_for(d)
    for o_dtype in (torch.float32, torch.bfloat16):
        o, lse = Banded((B, H, Nq, d), o_dtype), Banded((B, H, Nq), torch.float32)
        fa.forward_varlen(q, k, v, lq, lk, causal=causal, scale=scale, out=(o.t, lse.t))
        _check(("varlen fwd", causal, o_dtype), o, lse)
        dq = Banded((B, H, Nq, d), torch.float32)
        dk, dv = Banded((B, H, Nk, d), torch.float32), Banded((B, H, Nk, d), torch.float32)
        ws = Banded((B * H * Nq,), torch.float32)
        fa.backward_varlen(q, k, v, o.t, lse.t, do, lq, lk, causal=causal, scale=scale, workspace=ws.t,
                           out=(dq.t, dk.t, dv.t))
        _check(("varlen bwd", causal, o_dtype), dq, dk, dv, ws)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 20000), (3, 20000), (8, 129)])
def test_decode(Nq, Nk):
    B, H, d = 2, 4, 128
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=421 + Nk)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    o, lse = Banded((B, H, Nq, d), torch.float32), Banded((B, H, Nq), torch.float32)
    wsz = fa.fa_fwd_decode_workspace_bytes(B, H, Nq, Nk, d)
    ws = Banded((max(wsz // 4, 1),), torch.float32)
    fa.forward_decode(q, k, v, causal=True, workspace=ws.t, out=(o.t, lse.t))
    _check(("decode", Nq, Nk), o, lse, ws)
    # and with a padded batch (a sequence with no keys)
    lk = torch.tensor([Nk, 0], dtype=torch.int32, device="cuda")
    fa.forward_decode(q, k, v, None, lk, causal=True, workspace=ws.t, out=(o.t, lse.t))
    _check(("decode padded", Nq, Nk), o, lse, ws)


@pytest.mark.parametrize("N", [16, 144])
def test_fp8_forward(N):
    B, H, d = 1, 2, 128
    x8 = workloads.make_fp8_inputs(B, H, N, d, seed=431 + N)
    q8, k8, vt8 = (x8[n].cuda() for n in ("q", "k", "vt"))
    o, lse = Banded((B, H, N, d), torch.float32), Banded((B, H, N), torch.float32)
    fa.forward_fp8(q8, k8, vt8, causal=True, out=(o.t, lse.t))
    _check(("fp8", N), o, lse)


def test_masked_forward_backward():
    B, H, N, d = 2, 2, 129, 64
    inp = workloads.make_inputs(B, H, N, d, seed=441, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    gen = torch.Generator().manual_seed(443)
    bias = torch.randn(B, 1, N, N, generator=gen).to(torch.bfloat16).cuda()
    o, lse = Banded((B, H, N, d), torch.float32), Banded((B, H, N), torch.float32)
    fa.forward_bias(q, k, v, bias, causal=True, out=(o.t, lse.t))
    _check("bias fwd", o, lse)
    g = [Banded((B, H, N, d), torch.float32) for _ in range(3)]
    ws = Banded((B * H * N,), torch.float32)
    fa.backward_bias(q, k, v, o.t, lse.t, do, bias, causal=True, workspace=ws.t, out=tuple(x.t for x in g))
    _check("bias bwd", *g, ws)


def test_allocation_free_backward():
    B, H, N, d = 1, 3, 200, 128
    inp = workloads.make_inputs(B, H, N, d, seed=451, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    g = [Banded((B, H, N, d), torch.float32) for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    st = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                           g[0].t.data_ptr(), g[1].t.data_ptr(), g[2].t.data_ptr(), B, H, N, d, scale, 1, stream)
    assert st == 0, fa.fa_status_string(st)
    _check("noalloc", *g)


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_single_pass_backward(d, causal):
    """The single-pass backward adds every key tile's dQ share into dQ with
    reductions: none may land outside dQ (padded batch, ragged lengths)."""
    B, H, Nq, Nk = 3, 2, 300, 260
    sq, sk = [300, 0, 129], [260, 77, 200]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=461 + d)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    do = workloads.randn_bf16((B, H, Nq, d), 463 + d).cuda()
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(q, k, v, lq, lk, causal=causal)
    dq = Banded((B, H, Nq, d), torch.float32)
    dk, dv = Banded((B, H, Nk, d), torch.float32), Banded((B, H, Nk, d), torch.float32)
    ws = Banded((B * H * Nq,), torch.float32)
    fa.backward_single_pass(q, k, v, lse, do, None, lq, lk, causal=causal, workspace=ws.t, out=(dq.t, dk.t, dv.t))
    _check(("single pass", d, causal), dq, dk, dv, ws)
