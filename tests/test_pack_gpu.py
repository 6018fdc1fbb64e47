"""Bit-exact check of the device's FP32 -> 16-bit rounding (round to nearest, ties to
even) and of the word layout of a packed pair.

Every kernel of the library rounds FP32 to f16/bf16 with one routine (a paired
`cvt.rn` that puts the first value in the low half-word): the P operand of the PV
product, the attention epilogue and the combine's 16-bit output.  "Register fragments
and logical axes", section "Logical types and register packing", fixes that layout with
a worked word: packing the f16 pair (1, -2) gives 0xc0003c00.

The public `splitk_combine` reaches the routine with nothing else in the way: with one
partition, m* = lse_1, G = log2(2^0) + m* = m* and the partition weight 2^(lse_1 - G) is
exactly 1, so each output element is the FP32 input (times 1, plus +0) rounded to the
output type.  The expected bits come from the host: numpy's IEEE float16 conversion for
f16 and the integer round-to-nearest-even of `synth` (pinned to the page's word in
test_synth.py) for bf16.  Two cases differ from a bare conversion, by the arithmetic in
front of it: -0 leaves the accumulator as +0 (0 + (-0) = +0 under round to nearest), and
a NaN input comes out as some NaN (compared as a class, not by its payload)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ops = pytest.importorskip("online_softmax_gb300")

DEPTH = 128


def edge_values(dtype: str) -> np.ndarray:
    """Ties with even and odd kept mantissas, values just either side of a tie,
    subnormals of the target type, overflow to infinity, signed zeros, infinities."""
    f = np.float32
    ulp_f32 = lambda x: np.spacing(f(x))
    if dtype == "f16":
        t = 2.0 ** -11  # half an f16 ulp at 1
        base = [1.0 + t, 1.0 + 3 * t, 1.0 + t + 2.0 ** -20, 1.0 + t - 2.0 ** -20, 2.0 + 2 * t, 2.0 + 6 * t,
                2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -25 + 2.0 ** -40, 5 * 2.0 ** -26,
                2.0 ** -14 - 2.0 ** -25, 2.0 ** -14 - 2.0 ** -26, 2.0 ** -26,
                65504.0, 65519.0, 65520.0, 65536.0, 1e6, 0.1, 1.0 / 3.0]
    else:
        t = 2.0 ** -8  # half a bf16 ulp at 1
        base = [1.0 + t, 1.0 + 3 * t, 1.0 + t + 2.0 ** -20, 1.0 + t - 2.0 ** -20, 256.0 + 256 * t,
                2.0 ** -126, 2.0 ** -130, 2.0 ** -133 + 2.0 ** -141, 3 * 2.0 ** -134, 2.0 ** -149,
                float(np.finfo(np.float32).max), 3.3895313892515355e38, 3.3961e38, 0.1, 1.0 / 3.0]
    vals = np.array(base, dtype=np.float64)
    vals = np.concatenate([vals, -vals]).astype(f)
    extra = np.array([np.inf, -np.inf, 0.0, ulp_f32(1.0)], dtype=f)
    return np.concatenate([extra, vals])


def random_values(dtype: str, n: int, seed: int) -> np.ndarray:
    """Random FP32 bit patterns over the exponents that matter for the target type
    (every finite FP32 for bf16; |x| < 2^17 for f16, so its subnormals and overflow
    are in range), NaNs and infinities excluded."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    if dtype == "f16":
        exp = rng.integers(127 - 30, 127 + 17, n).astype(np.uint32)
        x = ((bits & np.uint32(0x807FFFFF)) | (exp << np.uint32(23))).view(np.float32)
    return x[np.isfinite(x)]


def device_round(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round x through splitk_combine with one partition; returns uint16 bits."""
    n = ((x.size + DEPTH - 1) // DEPTH) * DEPTH
    buf = np.zeros(n, dtype=np.float32)
    buf[: x.size] = x
    op = torch.from_numpy(buf.reshape(1, n // DEPTH, DEPTH)).cuda()
    lp = torch.full((1, n // DEPTH), 3.25, dtype=torch.float32, device="cuda")  # any finite LSE
    out = torch.empty((n // DEPTH, DEPTH), dtype={"f16": torch.float16, "bf16": torch.bfloat16}[dtype],
                      device="cuda")
    ops.splitk_combine(op, lp, out)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16).ravel()[: x.size]


def expected(x: np.ndarray, dtype: str) -> np.ndarray:
    with np.errstate(over="ignore"):  # overflow to infinity is one of the cases
        want = np.asarray(synth.round_to(x, dtype), dtype=np.uint16).copy()
    want[(x == 0)] = 0  # +0 and -0 both leave the accumulator as +0
    return want


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_edge_values_round_to_nearest_even(dtype):
    x = edge_values(dtype)
    got = device_round(x, dtype)
    want = expected(x, dtype)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "; ".join(f"{float(x[i])!r}: got {got[i]:#06x} want {want[i]:#06x}" for i in bad[:8])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_random_values_bit_exact(dtype):
    x = random_values(dtype, 1 << 20, 7 if dtype == "f16" else 8)
    got = device_round(x, dtype)
    want = expected(x, dtype)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {x.size} differ, e.g. {float(x[bad[0]])!r}: " \
                          f"{got[bad[0]]:#06x} vs {want[bad[0]]:#06x}"


def test_page_word_for_the_f16_pair():
    """("Register fragments and logical axes", Logical types and register packing): the
    f16 pair (1, -2) packs to the word 0xc0003c00, first value in the low half."""
    got = device_round(np.array([1.0, -2.0], dtype=np.float32), "f16")
    assert (int(got[0]) | (int(got[1]) << 16)) == 0xC0003C00


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nan_stays_nan(dtype):
    x = np.array([np.nan, -np.nan, 1.0], dtype=np.float32)
    got = device_round(x, dtype)
    exp_mask, man_mask = (0x7C00, 0x03FF) if dtype == "f16" else (0x7F80, 0x007F)
    for g in got[:2]:
        assert (g & exp_mask) == exp_mask and (g & man_mask) != 0, f"{g:#06x} is not a NaN"
    assert got[2] == synth.round_to(np.array([1.0], np.float32), dtype)[0]
