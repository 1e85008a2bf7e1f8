"""GPU parity away from unit-scale inputs: V, K and q multiplied by powers of
two, against the oracle with the output bound scaled alike (relative bound).

The tensor-core decode kernels take their PV operand P' = p * Delta_v (INT4)
or p * s_v (INT8) in fp16, with p <= 2^8 under the lazy softmax reference, and
the INT8 units take the query in fp16.  These cases put the fp16 operands near
both ends of their range:

- V x 2^-6: s_v a few times fp16's smallest normal value, so that P' of small
  probabilities is subnormal;
- V x 2^8: P' up to 2^8 * Delta_v, a few thousand, inside fp16;
- K x 2^-10: the INT8 key scales are fp16 subnormals;
- q x 2^-12 and q x 2^4: the query's fp16 form on the INT8 units, and nearly
  uniform or nearly one-hot attention.

Scaling a bf16 input by 2^e is exact, the quantization is scale-equivariant
while the metadata stays in fp16's normal range, and bf16 rounding of the
output commutes with the scaling, so the comparison is made on out * 2^-e
against ref * 2^-e with the unscaled rule (max-abs 2e-3, mean-abs 2e-4).

Beyond that range the append reports it: a V group whose Delta_v, or a
protected V whose s_v, exceeds 255.875 (P' could pass 65504) or is a nonzero
fp16 subnormal sets KV4_STATUS_V_RANGE; the bytes are stored as the oracle
stores them, and the CUDA-core kernel (fp32 throughout) still decodes them
within the tolerance.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from kv4_case import Case, compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


@pytest.fixture(autouse=True, params=[kv4.KV4_KERNEL_STREAM, kv4.KV4_KERNEL_MMA_SYNC,
                                      kv4.KV4_KERNEL_CUDA_CORE],
                ids=["stream", "mma", "cuda"])
def kernel(request):
    prev = kv4.kv4_set_decode_kernel(request.param)
    yield request.param
    kv4.kv4_set_decode_kernel(prev)


LENS = [700, 1500, 37, 3000, 1, 260]


@pytest.mark.parametrize("exps", [dict(v_exp=-6), dict(v_exp=8), dict(k_exp=-10),
                                  dict(q_exp=-12), dict(q_exp=4)],
                         ids=["v*2^-6", "v*2^8", "k*2^-10", "q*2^-12", "q*2^4"])
@pytest.mark.parametrize("g_", [32, 128])
def test_scaled_inputs_relative_parity(exps, g_):
    c = Case(LENS, S=4, R=64, g=g_, seed=41, **exps)
    gc = c.gpu()
    paged, side, st = c.oracle_cache()
    assert st == 0
    assert np.array_equal(gc.paged.cpu().numpy()[: paged.size], paged)
    assert np.array_equal(gc.side.cpu().numpy()[: side.size], side)
    out, lse = c.gpu_decode(gc)
    assert gc.read_status() == 0
    ref, rlse = c.oracle_decode()
    s = 2.0 ** -exps.get("v_exp", 0)
    compare_outputs({b: out[b] * s for b in range(c.B)}, lse,
                    {b: ref[b] * s for b in range(c.B)}, rlse, range(c.B), c.lens,
                    label=f"{exps} g={g_}")


@pytest.mark.parametrize("v_exp", [10, -10])
def test_v_beyond_fp16_operand_range_is_reported(v_exp, kernel):
    # V x 2^10: group ranges of 3.75 standard deviations reach 3840, Delta_v
    # > 255.875; V x 2^-10: max |V| of a token-head near 4.4e-3, so the
    # protected scales s_v = max|V| / 127 are fp16 subnormals
    c = Case([300, 90], S=4, R=16, g=32, seed=42, v_exp=v_exp)
    gc = c.gpu()
    assert gc.read_status() & kv4.KV4_STATUS_V_RANGE
    paged, side, st = c.oracle_cache()
    assert st == 0   # the encoding itself is the oracle's
    assert np.array_equal(gc.paged.cpu().numpy()[: paged.size], paged)
    assert np.array_equal(gc.side.cpu().numpy()[: side.size], side)
    if kernel == kv4.KV4_KERNEL_CUDA_CORE:   # fp32 throughout: still within the tolerance
        out, lse = c.gpu_decode(gc)
        ref, rlse = c.oracle_decode()
        s = 2.0 ** -v_exp
        compare_outputs({b: out[b] * s for b in range(c.B)}, lse,
                        {b: ref[b] * s for b in range(c.B)}, rlse, range(c.B), c.lens,
                        label=f"v*2^{v_exp} cuda-core")
    # inside the range: V x 2^8 and 2^-6 set nothing
    for e in (8, -6):
        assert Case([300, 90], S=4, R=16, g=32, seed=42, v_exp=e).gpu().read_status() == 0
