"""The GPU codec for quantised KV rows (q8_0 keys, q5_1 values) against the host codec and the
oracle: identical bytes and identical decoded f32 values on the same rows (the host codec is
itself byte-identical to the oracle, tests/test_kvq_host.py), and device-side errors recorded
instead of faulting."""
import numpy as np
import pytest
import torch

import quantized_transformer_decode_ql_gb300 as ql
from oracle import kvq

from gpu_util import lib
from test_kvq_host import rows_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["q8_0", "q5_1"])
@pytest.mark.parametrize("dim", [32, 128, 1024, 33, 100])
def test_device_codec_matches_host_and_oracle(fmt, dim):
    lib()
    x = rows_for(dim, dim + 1)
    rb = kvq.q8_row_bytes(dim) if fmt == "q8_0" else kvq.q5_row_bytes(dim)
    oq = kvq.quantize_q8_0 if fmt == "q8_0" else kvq.quantize_q5_1
    odq = kvq.dequantize_q8_0 if fmt == "q8_0" else kvq.dequantize_q5_1
    d_x = torch.from_numpy(x).cuda()
    d_out = torch.zeros((x.shape[0], rb), dtype=torch.uint8, device="cuda")
    ql.ql_kv_quantize_device(d_x, d_out, fmt)
    d_back = torch.zeros((x.shape[0], dim), dtype=torch.float32, device="cuda")
    ql.ql_kv_dequantize_device(d_out, d_back, fmt)
    torch.cuda.synchronize()
    ql.ql_check_device_error()
    got = d_out.cpu().numpy()
    want = oq(x)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
    host = ql.ql_kv_quantize_q8_0(x) if fmt == "q8_0" else ql.ql_kv_quantize_q5_1(x)
    assert np.array_equal(got, host)
    back = d_back.cpu().numpy()
    assert np.array_equal(back.view(np.uint32), odq(want, dim).view(np.uint32))


def test_device_codec_records_a_non_finite_value():
    lib()
    x = np.ones((3, 64), np.float32)
    x[2, 40] = np.inf
    d_x = torch.from_numpy(x).cuda()
    d_out = torch.zeros((3, kvq.q8_row_bytes(64)), dtype=torch.uint8, device="cuda")
    ql.ql_kv_quantize_device(d_x, d_out, "q8_0")
    with pytest.raises(ql.QLError) as e:
        ql.ql_check_device_error()
    assert e.value.status == ql.QL_EDEVICE and "non-finite" in str(e.value)
    ql.ql_check_device_error()   # read and cleared
    # the finite rows are still quantised exactly
    assert np.array_equal(d_out.cpu().numpy()[:2], kvq.quantize_q8_0(x[:2]))
