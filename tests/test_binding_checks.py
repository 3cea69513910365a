"""The Python binding hands the library raw pointers, so it checks every tensor it passes:
shape, dtype, contiguity and device of outputs, statistics and workspaces.  CPU tests of the
checking helpers, and GPU tests that wrongly shaped or placed tensors raise before any launch."""

import pytest
import torch

from exact_io_aware_fwd_gb300 import binding as fa

CPU = torch.device("cpu")


def test_want_accepts_exact_match_only():
    t = torch.empty(2, 3, dtype=torch.float32)
    assert fa._want(t, (2, 3), torch.float32, CPU, "t") is t
    with pytest.raises(ValueError):
        fa._want(t, (3, 2), torch.float32, CPU, "t")
    with pytest.raises(ValueError):
        fa._want(t, (2, 3), torch.bfloat16, CPU, "t")
    with pytest.raises(ValueError):
        fa._want(t.t(), (3, 2), torch.float32, CPU, "t")  # not contiguous
    with pytest.raises(ValueError):
        fa._want(None, (2, 3), torch.float32, CPU, "t")


def test_out_allocates_or_checks():
    t = fa._out(None, (4, 5), torch.bfloat16, CPU, "o")
    assert t.shape == (4, 5) and t.dtype == torch.bfloat16
    with pytest.raises(ValueError):
        fa._out(torch.empty(4, 6, dtype=torch.bfloat16), (4, 5), torch.bfloat16, CPU, "o")


def test_workspace_counts_bytes():
    ws, n = fa._workspace(torch.empty(100, dtype=torch.float32), 0, CPU)
    assert n == 400
    ws, n = fa._workspace(None, 1000, CPU)
    assert ws.dtype == torch.uint8 and ws.numel() == 1000 and n == 1000
    with pytest.raises(ValueError):
        fa._workspace(torch.empty(10, 10)[:, 0], 0, CPU)  # not contiguous


@pytest.mark.gpu
def test_wrong_outputs_raise_before_launch():
    import exact_io_aware_fwd_gb300 as pkg

    pkg.build()
    pkg.load_library()
    dev = torch.device("cuda", 0)
    B, H, N, d = 1, 2, 200, 64
    q, k, v, do = (torch.randn(B, H, N, d, device=dev).to(torch.bfloat16) for _ in range(4))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, out=torch.empty(B, H, N - 1, d, device=dev, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, lse=torch.empty(B, H, N, device=dev, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, lse=torch.empty(B, H, N))  # host memory
    o, lse = fa.fa_fwd(q, k, v)
    with pytest.raises(ValueError):
        fa.fa_bwd(q, k, v, o, do, lse[:, :1].contiguous())
    with pytest.raises(ValueError):
        fa.fa_bwd(q, k, v, o, do, lse, dq=torch.empty(B, H, N, d, device=dev))  # fp32
    # a workspace of any dtype is sized in bytes
    ws = torch.empty((fa.fa_bwd_workspace_size(B, H, N, d) + 3) // 4, device=dev,
                     dtype=torch.float32)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, workspace=ws)
    ref = fa.fa_bwd_deterministic(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    assert fa.fa_get_error() == fa.FA_OK
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    # grouped-query and variable-length wrappers check V, O, dO, LSE and the gradients too
    kg, vg = k[:, :1].contiguous(), v[:, :1].contiguous()
    with pytest.raises(ValueError):
        fa.fa_fwd_gqa(q, kg, v)
    og, lg = fa.fa_fwd_gqa(q, kg, vg)
    with pytest.raises(ValueError):
        fa.fa_bwd_gqa(q, kg, vg, og, do, lg, dk=torch.empty_like(k))
    qp, kp, vp = (t[0].transpose(0, 1).contiguous() for t in (q, k, v))  # [N, H, d]
    cu = torch.tensor([0, 120, N], dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(qp, kp, vp, cu.cpu(), 120)
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(qp, kp, vp, cu, 120, lse=torch.empty(N, H, device=dev))
