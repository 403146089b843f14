"""CPU tests of the Python binding's host logic: which C entry point
decode_attention calls for each kind of call, with which sizes, scale kind and
workspace size, and the dtype mapping of the tensors it passes.  The C entry
points are replaced by recorders, so nothing reaches a GPU."""
import pytest
import torch

import flash_decoding_attention_gb300 as fda


@pytest.fixture
def calls(monkeypatch):
    log = []

    def recorder(name):
        def f(*args, **kw):
            log.append((name, args, kw))
            return fda.FD_OK
        return f

    for name in ("fd_decode_attention", "fd_decode_attention_scaled",
                 "fd_decode_attention_multi", "fd_decode_attention_append"):
        monkeypatch.setattr(fda, name, recorder(name))
    monkeypatch.setattr(fda, "alloc_workspace",
                        lambda b, qh, kvh, d, dev=None: log.append(("ws", (b, qh, kvh, d), {}))
                        or torch.zeros(16, dtype=torch.uint8))
    return log


def _inputs(B=2, QH=8, KVH=2, D=64, rows=100, q_len=1, kv=torch.uint8):
    q = torch.zeros((B, QH, D) if q_len == 1 else (B, QH, q_len, D), dtype=torch.float16)
    k = torch.zeros((rows, KVH, D), dtype=kv)
    v = torch.zeros((rows, KVH, D), dtype=kv)
    seq = torch.tensor([5] * B, dtype=torch.int32)
    starts = torch.arange(B, dtype=torch.int32) * 10
    return q, k, v, seq, starts


def test_plain_call(calls):
    q, k, v, seq, starts = _inputs()
    out, lse = fda.decode_attention(q, k, v, seq, kv_start_idx=starts)
    names = [c[0] for c in calls]
    assert names == ["ws", "fd_decode_attention"]
    assert calls[0][1] == (2, 8, 2, 64)
    args = calls[1][1]
    assert args[6] == 100 and args[7:11] == (8, 2, 64, 0)      # kv_rows, QH, KVH, D, page
    assert abs(args[11] - 0.125) < 1e-12                       # default 1/sqrt(64)
    assert out.shape == q.shape and lse.shape == (2, 8)


@pytest.mark.parametrize("shape,kind", [((2,), fda.FD_SCALE_HEAD), ((100, 2), fda.FD_SCALE_TOKEN)])
def test_finer_scales_pick_the_kind(calls, shape, kind):
    q, k, v, seq, starts = _inputs()
    ks = torch.ones(shape)
    fda.decode_attention(q, k, v, seq, kv_start_idx=starts, k_scales=ks, v_scales=ks)
    name, args, _ = calls[-1]
    assert name == "fd_decode_attention_scaled" and args[14] == kind


def test_multi_token_queries(calls):
    q, k, v, seq, starts = _inputs(q_len=3)
    out, lse = fda.decode_attention(q, k, v, seq, kv_start_idx=starts)
    assert calls[0] == ("ws", (2, 8 * 3, 2, 64), {})            # workspace for QH * q_len rows
    name, args, _ = calls[-1]
    assert name == "fd_decode_attention_multi" and args[14] == fda.FD_SCALE_TENSOR
    assert out.shape == (2, 8, 3, 64) and lse.shape == (2, 8, 3)


@pytest.mark.parametrize("q_len", [1, 4])
def test_append_routes_to_the_fused_call(calls, q_len):
    q, k, v, seq, starts = _inputs(q_len=q_len)
    shape = (2, 2, 64) if q_len == 1 else (2, q_len, 2, 64)
    kn = torch.zeros(shape, dtype=torch.float16)
    pos = seq - q_len
    fda.decode_attention(q, k, v, seq, kv_start_idx=starts, k_new=kn, v_new=kn, positions=pos,
                         k_scales=torch.ones(100, 2), v_scales=torch.ones(100, 2))
    name, args, _ = calls[-1]
    assert name == "fd_decode_attention_append"
    assert args[1] is kn and args[7] is pos and args[17] == fda.FD_SCALE_TOKEN


def test_paged_sizes(calls):
    q = torch.zeros((3, 16, 128), dtype=torch.bfloat16)
    k = torch.zeros((40, 16, 1, 128), dtype=torch.uint8)           # 40 pages of 16 rows
    bt = torch.zeros((3, 8), dtype=torch.int32)
    seq = torch.tensor([1, 2, 3], dtype=torch.int32)
    fda.decode_attention(q, k, k, seq, block_table=bt)
    args = calls[-1][1]
    assert args[6] == 40 * 16 and args[10] == 16                    # kv_rows, page_size


def test_dtype_codes():
    assert fda._kv_dtype(torch.zeros(1, dtype=torch.int8)) == fda.FD_I8
    assert fda._kv_dtype(torch.zeros(1, dtype=torch.uint8)) == fda.FD_E4M3
    assert fda._kv_dtype(torch.zeros(1, dtype=torch.float8_e4m3fn)) == fda.FD_E4M3
    assert fda._kv_dtype(torch.zeros(1, dtype=torch.bfloat16)) == fda.FD_BF16
    assert fda._q_dtype(torch.zeros(1, dtype=torch.float16)) == fda.FD_F16
    with pytest.raises(ValueError):
        fda._kv_dtype(torch.zeros(1, dtype=torch.float32))
    with pytest.raises(ValueError):
        fda._q_dtype(torch.zeros(1, dtype=torch.int8))
    assert fda.DTYPE_CODES == {"f16": fda.FD_F16, "bf16": fda.FD_BF16, "e4m3": fda.FD_E4M3,
                               "i8": fda.FD_I8}
