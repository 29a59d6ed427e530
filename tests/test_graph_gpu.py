"""The entry points under CUDA graph capture: a Linear forward + backward (row-wise and tensorwise
recipes) and a grouped GEMM are captured once into a graph and replayed; every output must be
bit-identical to the same calls run eagerly (the kernels are deterministic: fixed accumulation
order per tile, commutative integer max for amax). Capture needs no allocation, host
synchronisation or host-side read of device data inside the library: workspaces come from the
caller, offsets stay on the device."""
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, upload_codes, upload_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _linear_buffers(fp8, M, K, N, gran, wgrad):
    d = "cuda"
    x, w, dy = W.linear_inputs(M, K, N, seed=21, device=d, outliers=True)
    e4 = torch.float8_e4m3fn
    tens = gran == fp8.GRAN_TENSOR
    b = dict(
        x=x, w=w, dy=dy,
        x_q=torch.empty((M, K), dtype=e4, device=d), w_q=torch.empty((N, K), dtype=e4, device=d),
        x_inv=torch.empty(1 if tens else M, device=d), w_inv=torch.empty(1 if tens else N, device=d),
        xt_q=torch.empty((K, M), dtype=e4, device=d) if tens else None,
        wt_q=torch.empty((K, N), dtype=e4, device=d) if tens else None,
        y=torch.empty((M, N), dtype=torch.bfloat16, device=d),
        dx=torch.empty((M, K), dtype=torch.bfloat16, device=d),
        dw=torch.empty((N, K), dtype=torch.bfloat16, device=d),
        ws_f=torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_FWD, M, K, N, gran), 16), dtype=torch.uint8, device=d),
        ws_b=torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, gran, wgrad), 16), dtype=torch.uint8,
                         device=d),
        st=torch.zeros(1, dtype=torch.int32, device=d),
    )
    b["saved"] = fp8.make_saved(b["x_q"], b["x_inv"], b["w_q"], b["w_inv"], b["xt_q"], b["wt_q"])
    return b


def _linear_step(fp8, b, gran, wgrad):
    fp8.fp8_linear_fwd(b["x"], b["w"], gran, fp8.MM_FAST_ACCUM, b["y"], b["saved"], b["ws_f"], b["st"])
    fp8.fp8_linear_bwd(b["dy"], b["saved"], b["x"], b["w"], gran, wgrad, b["dx"], b["dw"], b["ws_b"], b["st"])


def _snapshot(b, keys):
    return {k: b[k].clone() for k in keys if b[k] is not None}


@pytest.mark.parametrize("gran_name,wgrad", [("GRAN_ROW", 1), ("GRAN_ROW", 0), ("GRAN_TENSOR", 0)])
def test_linear_graph_replay_matches_eager(fp8, gran_name, wgrad):
    gran = getattr(fp8, gran_name)
    M, K, N = 2048, 1024, 1536  # large enough for the CTA-pair GEMMs
    b = _linear_buffers(fp8, M, K, N, gran, wgrad)
    keys = ["x_q", "x_inv", "w_q", "w_inv", "xt_q", "wt_q", "y", "dx", "dw"]
    _linear_step(fp8, b, gran, wgrad)
    torch.cuda.synchronize()
    eager = _snapshot(b, keys)
    for k in ("y", "dx", "dw"):
        b[k].fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        _linear_step(fp8, b, gran, wgrad)  # a warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for k in ("y", "dx", "dw"):
        b[k].fill_(float("nan"))
    with torch.cuda.graph(g):
        _linear_step(fp8, b, gran, wgrad)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(b["st"].item()) == 0
    for k, v in eager.items():
        assert torch.equal(b[k].view(torch.uint8) if b[k].dtype.is_floating_point and b[k].element_size() == 1 else b[k],
                           v.view(torch.uint8) if v.dtype.is_floating_point and v.element_size() == 1 else v), k


def test_grouped_graph_replay_matches_eager(fp8):
    counts = [300, 0, 1500, 7, 260]
    E, M, N, K = len(counts), sum(counts), 512, 256
    A = W.normal_bf16((M, K), 1.0, 3)
    Wt = W.normal_bf16((E, N, K), 0.02, 4)
    ca, ia = oracle.quantize_rows(bits(A), oracle.E4M3)
    cw, iw = oracle.quantize_rows(bits(Wt).reshape(E * N, K), oracle.E4M3)
    a, w = upload_codes(ca, oracle.E4M3), upload_codes(cw.reshape(E, N, K), oracle.E4M3)
    sa, sw = upload_f32(ia), upload_f32(iw.reshape(E, N))
    ends = torch.from_numpy(W.ends_from_counts(counts)).cuda()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8.fp8_grouped_mm(a, w, ends, sa, sw, out, fp8.GROUPED_JAGGED_M)
    torch.cuda.synchronize()
    eager = out.clone()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp8.fp8_grouped_mm(a, w, ends, sa, sw, out, fp8.GROUPED_JAGGED_M)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("gran_name,wgrad_name", [("GRAN_MX", "WGRAD_FP8"), ("GRAN_BLOCK_1x128", "WGRAD_BF16")])
def test_mx_and_blockwise_linear_graph_replay(fp8, gran_name, wgrad_name):
    """The MX and blockwise Linear forward + backward captured into one graph and replayed:
    bit-identical to the eager calls."""
    gran, wgrad = getattr(fp8, gran_name), getattr(fp8, wgrad_name)
    M, K, N = 1024, 512, 768
    x, w, dy = W.linear_inputs(M, K, N, seed=22, device="cuda", outliers=True)
    saved, bufs = fp8.linear_saved_alloc(M, K, N, gran, keep_xt=wgrad == fp8.WGRAD_FP8)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, gran, wgrad), 16), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        fp8.fp8_linear_fwd(x, w, gran, fp8.MM_FAST_ACCUM, y, saved, None, st)
        fp8.fp8_linear_bwd(dy, saved, x, w, gran, wgrad, dx, dw, ws, st)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (y, dx, dw)] + [b.clone() for b in bufs if b is not None]
    for t in (y, dx, dw):
        t.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in (y, dx, dw):
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    now = [y, dx, dw] + [b for b in bufs if b is not None]
    for a, b in zip(now, eager):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
