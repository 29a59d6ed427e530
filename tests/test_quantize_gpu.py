"""GPU parity of the fused quantize kernels against the CPU oracle: FP8 codes and fp32 inverse
scales must be bit-identical ("FP8 Training: Quantization, Autograd, Torchao", section 2).

Shapes span several tiles, ragged tails (rows not a multiple of the row tile, columns not a
multiple of the 64-column strip), tiny and empty inputs, and rows built to hit exact FP8 ties,
FP8 subnormals, a huge outlier, all zeros and negative zeros."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, codes, f32_bits, special_rows

pytestmark = pytest.mark.gpu

FMTS = [(oracle.E4M3, 3, 448.0), (oracle.E5M2, 4, 57344.0)]  # (oracle fmt, library dtype, max)


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _input(R, C, seed, fmax, std=1.0):
    x = W.normal_bf16((R, C), std, seed)
    if R >= 8:
        sp = special_rows(C, fmax)
        x[1:1 + sp.shape[0]] = sp
    return x


@pytest.mark.parametrize("R,C", [(1, 8), (5, 24), (300, 512), (257, 4096), (64, 14336), (33, 7168), (7, 65536)])
@pytest.mark.parametrize("fi", [0, 1])
def test_rowwise(fp8, R, C, fi):
    ofmt, dt, fmax = FMTS[fi]
    x = _input(R, C, 100 + R, fmax)
    q, _, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_ROW, dt)
    torch.cuda.synchronize()
    q_ref, inv_ref = oracle.quantize_rows(bits(x), ofmt)
    assert np.array_equal(codes(q), q_ref)
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


def test_rowwise_3d_and_empty(fp8):
    x = W.normal_bf16((3, 40, 96), 0.02, 7)
    q, _, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_ROW, fp8.DT_E4M3)
    q_ref, inv_ref = oracle.quantize_rows(bits(x).reshape(120, 96), oracle.E4M3)
    assert np.array_equal(codes(q).reshape(120, 96), q_ref)
    assert np.array_equal(f32_bits(inv).reshape(-1), inv_ref.view(np.uint32))
    x0 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q0, _, inv0 = fp8.quantize_alloc(x0, fp8.GRAN_ROW, fp8.DT_E4M3)
    assert q0.numel() == 0


def _every_amax(rows_per_pattern_cols: int):
    """One row per non-negative finite bf16 pattern p (0x0000 .. 0x7F7F): p itself, its negation,
    then values |v| <= p (p with lower mantissa bits cleared, and zeros), so that the row's amax
    is exactly p and every scale the format can take is hit once."""
    p = np.arange(0x7F80, dtype=np.uint16)
    x = np.zeros((p.size, rows_per_pattern_cols), np.uint16)
    x[:, 0] = p
    x[:, 1] = p | 0x8000
    x[:, 2] = p & 0xFFF0
    x[:, 3] = (p & 0xFF80) | 0x8000
    return x


@pytest.mark.parametrize("fi", [0, 1])
def test_scale_every_bf16_amax(fp8, fi):
    """Exhaustive check of the scale step: the row scales (and, transposed, the column scales)
    for every finite non-negative bf16 amax, below eps, subnormal, up to the largest bf16,
    bit-identical with the oracle's fp64 division."""
    ofmt, dt, _ = FMTS[fi]
    xb = _every_amax(16)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    q, _, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_ROW, dt)
    q_ref, inv_ref = oracle.quantize_rows(xb, ofmt)
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))
    assert np.array_equal(codes(q), q_ref)
    xt = x.T.contiguous()  # [16, 32640]: one pattern per column
    _, qt, invc = fp8.quantize_alloc(xt.cuda(), fp8.GRAN_COL, dt)
    qc_ref, invc_ref = oracle.quantize_cols(np.ascontiguousarray(xb.T), ofmt)
    assert np.array_equal(f32_bits(invc), invc_ref.view(np.uint32))
    assert np.array_equal(codes(qt), qc_ref.T)


@pytest.mark.parametrize("R,C", [(16, 8), (256, 512), (130 * 16, 200), (1024, 1000)])
@pytest.mark.parametrize("fi", [0, 1])
def test_tensorwise_dual_output(fp8, R, C, fi):
    ofmt, dt, fmax = FMTS[fi]
    x = _input(R, C, 200 + R, fmax)
    q, qt, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_TENSOR, dt, layout=fp8.LAYOUT_BOTH)
    torch.cuda.synchronize()
    q_ref, inv_ref = oracle.quantize_tensor(bits(x), ofmt)
    assert np.array_equal(codes(q), q_ref)
    assert np.array_equal(codes(qt), q_ref.T)  # column-major output = transpose of the row-major codes
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))
    # single-layout calls agree with the dual output
    q1, _, _ = fp8.quantize_alloc(x.cuda(), fp8.GRAN_TENSOR, dt, layout=fp8.LAYOUT_ROW_MAJOR)
    _, qt1, _ = fp8.quantize_alloc(x.cuda(), fp8.GRAN_TENSOR, dt, layout=fp8.LAYOUT_COL_MAJOR)
    assert np.array_equal(codes(q1), q_ref) and np.array_equal(codes(qt1), q_ref.T)


@pytest.mark.parametrize("R,C,layout", [(4096, 4096, "both"), (4112, 4160, "both"), (4112, 4104, "col"),
                                         (6144, 2112, "col"), (16, 64, "both")])
def test_tensorwise_stash_shapes(fp8, R, C, layout):
    """The tensorwise kernel that keeps each SM's last 8 tiles of 128 x 64 on chip: enough tiles
    that its ring wraps (2048+ tiles over 152 SMs, 13+ per SM), ragged last tile rows and columns,
    the column-major output alone, a single tile."""
    ofmt, dt, fmax = FMTS[0]
    x = _input(R, C, 300 + R + C, fmax)
    lay = fp8.LAYOUT_BOTH if layout == "both" else fp8.LAYOUT_COL_MAJOR
    q, qt, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_TENSOR, dt, layout=lay)
    torch.cuda.synchronize()
    q_ref, inv_ref = oracle.quantize_tensor(bits(x), ofmt)
    assert np.array_equal(codes(qt), q_ref.T)
    if layout == "both":
        assert np.array_equal(codes(q), q_ref)
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


@pytest.mark.parametrize("R,C", [(16, 8), (512, 64), (1040, 200), (8192, 136), (9216, 72), (20480, 64),
                                 (2048, 2048), (1040, 4096)])
@pytest.mark.parametrize("fi", [0, 1])
def test_colwise_transposed(fp8, R, C, fi):
    """Column scales with column-major output; R = 20480 takes the two-pass path (groups above
    8 x 1024 rows)."""
    ofmt, dt, fmax = FMTS[fi]
    # column-gain input as in the backward-operand workload
    x = W.column_gain_bf16((R, C), 1e-3, -2, 2, 301 + R)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, qt, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_COL, dt, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_ref, inv_ref = oracle.quantize_cols(bits(x), ofmt)
    assert np.array_equal(codes(qt), q_ref.T)
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


def test_colwise_special_columns(fp8):
    """The special patterns run down the columns (ties at scale 1, subnormals, outliers, zeros)."""
    for ofmt, dt, fmax in FMTS:
        sp = special_rows(32, fmax).T  # [32 rows, 5 pattern columns]
        x = torch.cat([sp, W.normal_bf16((32, 3), 1.0, 3)], 1).contiguous()
        _, qt, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_COL, dt)
        q_ref, inv_ref = oracle.quantize_cols(bits(x), ofmt)
        assert np.array_equal(codes(qt), q_ref.T)
        assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


@pytest.mark.parametrize("B,R,C", [(3, 64, 96), (4, 7168 // 8, 256), (2, 16, 8), (40, 256, 200), (8, 1040, 512)])
def test_colwise_batched_3d(fp8, B, R, C):
    """Per-expert column scales of a 3-D weight [E, K, N] (amax over K for each (e, n))."""
    x = W.normal_bf16((B, R, C), 0.02, 400 + B)
    _, qt, inv = fp8.quantize_alloc(x.cuda(), fp8.GRAN_COL, fp8.DT_E4M3)
    q_ref, inv_ref = oracle.quantize_cols(bits(x), oracle.E4M3)
    assert np.array_equal(codes(qt), np.transpose(q_ref, (0, 2, 1)))
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


def _segpad(q_ref, ends, P):
    """Oracle codes [R, C] -> the segment-padded column-major layout [C, P]."""
    R, C = q_ref.shape
    out = np.zeros((C, P), np.uint8)
    prev, pos = 0, 0
    for e in ends:
        n = e - prev
        out[:, pos:pos + n] = q_ref[prev:e].T
        pos += -(-n // 128) * 128
        prev = e
    return out, pos


@pytest.mark.parametrize("counts", [[100, 0, 37, 500, 1], [0, 0, 64], [300, 0], [9000, 5, 0, 11000],
                                    list(W.llama4_counts(0) // 4), list(W.random_counts(3000, 40, 5, n_empty=9)),
                                    [0] * 7 + [1000] + [0] * 9,
                                    [31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129, 224, 225, 255, 256, 257, 511]])
@pytest.mark.parametrize("fi", [0, 1])
def test_jagged_colwise(fp8, counts, fi):
    """Column scales per segment, written into the segment-padded column-major layout; a segment's
    last, partial 256-row tile loads only the 32-row boxes holding its rows (the last case puts
    segment tails on both sides of each 32-row boundary)."""
    ofmt, dt, fmax = FMTS[fi]
    counts = [int(c) for c in counts]
    R = sum(counts)
    C = 72
    x = W.normal_bf16((R, C), 1e-3, 500 + R)
    ends = W.ends_from_counts(counts)
    P = fp8.fp8_jagged_padded_rows(R, len(counts))
    if fi == 1:  # a pitch that is a multiple of 16 but not of 128 bytes is accepted too
        P = W.ceil_div(R + 127 * len(counts), 16) * 16
        P += 16 if P % 128 == 0 else 0
    canary = torch.full((C, P), 0x5A, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn if dt == 3 else torch.float8_e5m2)
    inv = torch.empty((len(counts), C), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_COL, dt, fp8.LAYOUT_COL_MAJOR, None, canary, inv,
                     torch.from_numpy(ends).cuda(), fp8.col_workspace(len(counts), C, R, "cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_ref, inv_ref = oracle.quantize_jagged_cols(bits(x), ends, ofmt)
    ref, used = _segpad(q_ref, ends, P)
    got = codes(canary)
    assert np.array_equal(got[:, :used], ref[:, :used])  # data and zero padding
    assert np.all(got[:, used:] == 0x5A)  # nothing written past the last padded segment
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


@pytest.mark.parametrize("counts", [list(W.llama4_counts(1) // 2), [700, 0, 1300, 5, 0, 2100]])
def test_jagged_colwise_wide(fp8, counts):
    """Segment columns with many 256-row x 64-column work units per CTA (C = 1024)."""
    counts = [int(c) for c in counts]
    R, C = sum(counts), 1024
    x = W.normal_bf16((R, C), 1e-2, 600 + R)
    ends = W.ends_from_counts(counts)
    P = fp8.fp8_jagged_padded_rows(R, len(counts))
    out = torch.full((C, P), 0x5A, dtype=torch.uint8, device="cuda").view(torch.float8_e5m2)
    inv = torch.empty((len(counts), C), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_COL, fp8.DT_E5M2, fp8.LAYOUT_COL_MAJOR, None, out, inv,
                     torch.from_numpy(ends).cuda(), fp8.col_workspace(len(counts), C, R, "cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_ref, inv_ref = oracle.quantize_jagged_cols(bits(x), ends, oracle.E5M2)
    ref, used = _segpad(q_ref, ends, P)
    got = codes(out)
    assert np.array_equal(got[:, :used], ref[:, :used])
    assert np.all(got[:, used:] == 0x5A)
    assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


def test_jagged_colwise_segment_limit(fp8):
    """The most segments a column quantize takes (2048: its per-segment prefix arrays live in
    shared memory), most of them a few rows long or empty; one segment more is rejected."""
    C = 16
    for E, ok in ((2048, True), (2049, False)):
        counts = [int(c) for c in W.random_counts(6000, E, 7, n_empty=E // 4)]
        R = sum(counts)
        x = W.normal_bf16((R, C), 1.0, 700 + E)
        ends = W.ends_from_counts(counts)
        P = fp8.fp8_jagged_padded_rows(R, E)
        out = torch.full((C, P), 0x5A, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
        inv = torch.empty((E, C), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (x.cuda(), fp8.GRAN_COL, fp8.DT_E4M3, fp8.LAYOUT_COL_MAJOR, None, out, inv,
                torch.from_numpy(ends).cuda(), fp8.col_workspace(E, C, R, "cuda"))
        if not ok:
            with pytest.raises(fp8.Fp8Error) as e:
                fp8.fp8_quantize(*args, status=st)
            assert e.value.code == 2
            continue
        fp8.fp8_quantize(*args, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        q_ref, inv_ref = oracle.quantize_jagged_cols(bits(x), ends, oracle.E4M3)
        ref, used = _segpad(q_ref, ends, P)
        got = codes(out)
        assert np.array_equal(got[:, :used], ref[:, :used])
        assert np.all(got[:, used:] == 0x5A)
        assert np.array_equal(f32_bits(inv), inv_ref.view(np.uint32))


def test_jagged_bad_offsets_sets_status(fp8):
    x = W.normal_bf16((64, 8), 1.0, 9).cuda()
    P = fp8.fp8_jagged_padded_rows(64, 3)
    out = torch.zeros((8, P), dtype=torch.float8_e4m3fn, device="cuda")
    inv = torch.zeros((3, 8), dtype=torch.float32, device="cuda")
    for bad in ([10, 5, 64], [10, 20, 63]):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp8.fp8_quantize(x, fp8.GRAN_COL, fp8.DT_E4M3, fp8.LAYOUT_COL_MAJOR, None, out, inv,
                         torch.tensor(bad, dtype=torch.int32, device="cuda"), fp8.col_workspace(3, 8, 100, "cuda"), status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == fp8.DEV_BAD_OFFSETS


def test_argument_errors(fp8):
    x = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")  # C % 8 != 0
    inv = torch.zeros(16, dtype=torch.float32, device="cuda")
    q = torch.zeros((16, 12), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_quantize(x, fp8.GRAN_ROW, fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR, q, None, inv)
    assert e.value.code == 3
    x = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:  # wrong inv length
        fp8.fp8_quantize(x, fp8.GRAN_ROW, fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR,
                         torch.zeros((16, 16), dtype=torch.float8_e4m3fn, device="cuda"), None, inv[:3])
    assert e.value.code == 1
    with pytest.raises(fp8.Fp8Error) as e:  # column granularity without its per-column workspace
        fp8.fp8_quantize(x, fp8.GRAN_COL, fp8.DT_E4M3, fp8.LAYOUT_COL_MAJOR, None,
                         torch.zeros((16, 16), dtype=torch.float8_e4m3fn, device="cuda"), inv)
    assert e.value.code == 4
    with pytest.raises(fp8.Fp8Error) as e:  # tensor granularity without workspace
        fp8.fp8_quantize(x, fp8.GRAN_TENSOR, fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR,
                         torch.zeros((16, 16), dtype=torch.float8_e4m3fn, device="cuda"), None, inv[:1])
    assert e.value.code == 4
