"""Host-side checks of the Python binding (no GPU): every buffer must hold the
elements its entry point touches, code tensors may be uint8 or
float8_e4m3fn, and nothing reaches the library until the checks pass.

On CPU tensors a call whose sizes and dtypes are right stops at the CUDA
device check, which shows that the size checks let it through; the shapes
below include those the GPU tests and the benchmark use."""
import pytest
import torch

from fp8_w8a8_quantized_group_gb300 import _lib, ops

BF16, F32, U8, I32 = torch.bfloat16, torch.float32, torch.uint8, torch.int32
NOT_CUDA = "must be a CUDA tensor"


@pytest.fixture(autouse=True)
def _no_library(monkeypatch):
    """Any call that got past the checks would load the library: make that an error."""
    def refuse():
        raise AssertionError("the library was reached before the argument checks failed")
    monkeypatch.setattr(_lib, "load", refuse)


def e(*shape, dtype=U8):
    return torch.empty(shape, dtype=dtype)


def _block_gemm_args(M, N, K, E=1):
    qw = e(E, N, K) if E > 1 else e(N, K)
    sw = e(E, -(-N // 128), K // 128, dtype=F32) if E > 1 else e(-(-N // 128), K // 128, dtype=F32)
    return dict(qa=e(M, K), sa=e(K // 128, M, dtype=F32), qw=qw, sw=sw, y=e(M, N, dtype=BF16))


@pytest.mark.parametrize("M,N,K", [(16, 28672, 4096), (1, 4096, 14336), (300, 272, 640), (2048, 6144, 4096)])
def test_block_gemm_sizes_pass(M, N, K):
    a = _block_gemm_args(M, N, K)
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"], a["sw"], a["y"])


def test_grouped_sizes_pass():
    a = _block_gemm_args(8192, 2048, 7168, E=8)
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"], a["sw"], a["y"], num_groups=8,
                           group_offsets=e(9, dtype=I32))


@pytest.mark.parametrize("which,shrink", [("sa", 1), ("qw", 1), ("sw", 1), ("y", 1)])
def test_block_gemm_refuses_a_short_buffer(which, shrink):
    a = _block_gemm_args(40, 256, 512)
    t = a[which]
    # y fixes N by its shape, so a short y has a row too few
    a[which] = e(39, 256, dtype=BF16) if which == "y" else t.flatten()[: t.numel() - shrink]
    with pytest.raises(ValueError, match=f"^{which}: has"):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"], a["sw"], a["y"])


def test_grouped_refuses_dense_weights_and_short_offsets():
    a = _block_gemm_args(64, 256, 512, E=4)
    with pytest.raises(ValueError, match="^qw: has"):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"][0], a["sw"], a["y"], num_groups=4,
                           group_offsets=e(5, dtype=I32))
    with pytest.raises(ValueError, match="^sw: has"):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"], a["sw"][0], a["y"], num_groups=4,
                           group_offsets=e(5, dtype=I32))
    with pytest.raises(ValueError, match="^group_offsets: has"):
        ops.fp8_block_gemm(a["qa"], a["sa"], a["qw"], a["sw"], a["y"], num_groups=4,
                           group_offsets=e(4, dtype=I32))


def test_larger_buffers_and_float8_codes_pass():
    """A buffer may be larger than the call needs (e.g. with guard bytes), and
    codes may come as float8_e4m3fn."""
    a = _block_gemm_args(40, 256, 512)
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_block_gemm(a["qa"].view(torch.float8_e4m3fn), a["sa"], a["qw"].view(torch.float8_e4m3fn),
                           a["sw"], e(41, 256, dtype=BF16))


def test_wrong_dtype_is_a_type_error():
    a = _block_gemm_args(40, 256, 512)
    with pytest.raises(TypeError, match="^sa: expected torch.float32"):
        ops.fp8_block_gemm(a["qa"], a["sa"].to(torch.float64), a["qw"], a["sw"], a["y"])
    with pytest.raises(TypeError, match="^qa: expected torch.uint8 or torch.float8_e4m3fn"):
        ops.fp8_block_gemm(a["qa"].to(torch.int8), a["sa"], a["qw"], a["sw"], a["y"])


def test_tensor_gemm_sizes():
    M, N, K = 16, 8192, 8192
    args = [e(M, K), e(1, dtype=F32), e(N, K), e(1, dtype=F32), e(M, N, dtype=BF16)]
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_tensor_gemm(*args)
    for i, name in [(1, "sa"), (3, "sw")]:
        bad = list(args)
        bad[i] = e(0, dtype=F32)
        with pytest.raises(ValueError, match=f"^{name}: has"):
            ops.fp8_tensor_gemm(*bad)
    bad = list(args)
    bad[2] = e(N - 1, K)
    with pytest.raises(ValueError, match="^qw: has"):
        ops.fp8_tensor_gemm(*bad)


def test_block_linear_sizes():
    M, N, K = 5, 19584, 8320
    args = [e(M, K, dtype=BF16), e(M, K), e(K // 128, M, dtype=F32), e(N, K), e(-(-N // 128), K // 128, dtype=F32),
            e(M, N, dtype=BF16)]
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_block_linear(*args)
    for i, name in enumerate(["x", "qa", "sa", "qw", "sw", "y"]):
        if name == "x":
            continue  # M and K come from x's shape
        bad = list(args)
        bad[i] = e(M - 1, N, dtype=BF16) if name == "y" else args[i].flatten()[:-1]
        with pytest.raises(ValueError, match=f"^{name}: has"):
            ops.fp8_block_linear(*bad)


def test_quantizer_sizes():
    M, K = 17, 384
    x = e(M, K, dtype=BF16)
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_quant_act_group(x, e(M, K), e(K // 128, M, dtype=F32))
    with pytest.raises(ValueError, match="^q: has"):
        ops.fp8_quant_act_group(x, e(M - 1, K), e(K // 128, M, dtype=F32))
    with pytest.raises(ValueError, match="^scales: has"):
        ops.fp8_quant_act_group(x, e(M, K), e(K // 128, M - 1, dtype=F32))

    N = 130
    w = e(N, 256, dtype=BF16)
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_quant_weight_block(w, e(N, 256), e(2, 2, dtype=F32))
    with pytest.raises(ValueError, match="^scales: has"):
        ops.fp8_quant_weight_block(w, e(N, 256), e(1, 2, dtype=F32))  # the ragged block row needs a scale too

    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_quant_per_tensor(x, e(M, K), e(1, dtype=F32), False)
    with pytest.raises(ValueError, match="^scale: has"):
        ops.fp8_quant_per_tensor(x, e(M, K), e(0, dtype=F32), True)


def test_zero_rows_need_no_buffers():
    """M = 0 is a valid call that touches nothing."""
    with pytest.raises(ValueError, match=NOT_CUDA):
        ops.fp8_quant_act_group(e(0, 256, dtype=BF16), e(0), e(0, dtype=F32))
