"""CPU checks of the C ABI: the library builds and loads, exports every
function include/fd_attention.h declares, and rejects bad arguments on the
host before any launch (these calls never reach the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd_attention.h")


@pytest.fixture(scope="module")
def fda():
    from flash_decoding_attention_gb300 import build
    build.build()
    import flash_decoding_attention_gb300 as m
    m.load_library()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["fd_decode_attention", "fd_workspace_bytes", "fd_check_device_error",
              "fd_status_string", "fd_debug_read_plan", "fd_debug_gather_kv"]:
        assert n in names


def test_library_exports_every_declared_symbol(fda):
    lib = ctypes.CDLL(fda.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(fda.EXPORTED) == declared_functions()


def test_status_strings(fda):
    for st in range(7):
        assert fda.fd_status_string(st)
    assert fda.fd_status_string(99) == "unknown status"


def _call(fda, **over):
    """fd_decode_attention with fake (never dereferenced) device pointers."""
    lib = fda.load_library()
    a = dict(q=0x1000, k=0x2000, v=0x3000, kv_start=0x4000, bt=None, bt_stride=0,
             seq_len=0x5000, kv_rows=100, batch=2, qh=8, kvh=2, d=128, page=0,
             ss=0.125, ks=1.0, vs=1.0, qdt=0, kvdt=0, out=0x6000, lse=0x7000, ws=0x8000,
             wsb=1 << 20, stream=None)
    a.update(over)
    return lib.fd_decode_attention(a["q"], a["k"], a["v"], a["kv_start"], a["bt"], a["bt_stride"],
                                   a["seq_len"], a["kv_rows"], a["batch"], a["qh"], a["kvh"],
                                   a["d"], a["page"], a["ss"], a["ks"], a["vs"], a["qdt"],
                                   a["kvdt"], a["out"], a["lse"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(q=None), 1),
    (dict(k=None), 1),
    (dict(seq_len=None), 1),
    (dict(out=None), 1),
    (dict(ws=None), 1),
    (dict(bt=0x9000, bt_stride=4, page=16), 1),          # both layouts given
    (dict(kv_start=None), 1),                              # neither layout
    (dict(batch=0), 1),
    (dict(qh=6, kvh=4), 1),                                # heads not divisible
    (dict(d=96), 2),                                       # unsupported head_dim
    (dict(kv_start=None, bt=0x9000, bt_stride=4, page=48, kv_rows=96), 2),   # page not pow2
    (dict(kv_start=None, bt=0x9000, bt_stride=0, page=16, kv_rows=96), 1),   # bad stride
    (dict(kv_start=None, bt=0x9000, bt_stride=4, page=16, kv_rows=100), 1),  # rows % page
    (dict(kv_rows=0), 1),
    (dict(qdt=2), 1),                                      # q cannot be e4m3
    (dict(qdt=3), 1),                                      # q cannot be int8
    (dict(kvdt=4), 1),                                     # unknown cache format
    (dict(qdt=0, kvdt=1), 2),                              # f16 q with bf16 cache
    (dict(ss=float("nan")), 1),
    (dict(q=0x1001), 1),                                   # misaligned q
    (dict(ws=0x8010), 1),                                  # misaligned workspace
])
def test_host_validation(fda, over, status):
    assert _call(fda, **over) == status


def _call_scaled(fda, kind, k_scales, v_scales, kvdt):
    """fd_decode_attention_scaled with fake pointers; only argument errors
    are asked for, so nothing is ever launched."""
    lib = fda.load_library()
    return lib.fd_decode_attention_scaled(0x1000, 0x2000, 0x3000, 0x4000, None, 0, 0x5000, 100, 2,
                                          8, 2, 128, 0, 0.125, 1.0, 1.0, kind, k_scales, v_scales,
                                          0, kvdt, 0x6000, 0x7000, 0x8000, 1 << 20, None)


@pytest.mark.parametrize("kind,ks,vs,kvdt,status", [
    (3, 0xA000, 0xB000, 2, 1),          # unknown scale kind
    (1, None, 0xB000, 2, 1),            # missing K scales
    (2, 0xA000, None, 3, 1),            # missing V scales
    (2, 0xA002, 0xB000, 3, 1),          # misaligned K scales
    (1, 0xA000, 0xB000, 0, 2),          # finer scales on an f16 cache
    (2, 0xA000, 0xB000, 1, 2),          # finer scales on a bf16 cache
])
def test_scaled_host_validation(fda, kind, ks, vs, kvdt, status):
    assert _call_scaled(fda, kind, ks, vs, kvdt) == status


def _call_append(fda, **over):
    """fd_append_kv with fake pointers; only argument errors are asked for."""
    a = dict(kn=0x1000, vn=0x2000, k=0x3000, v=0x4000, kv_start=0x5000, bt=None, bt_stride=0,
             pos=0x6000, kv_rows=100, batch=2, n_new=1, kvh=2, d=128, page=0, ks=1.0, vs=1.0,
             kind=0, kss=None, vss=None, ndt=0, kvdt=2, ws=0x8000, wsb=256)
    a.update(over)
    return fda.load_library().fd_append_kv(
        a["kn"], a["vn"], a["k"], a["v"], a["kv_start"], a["bt"], a["bt_stride"], a["pos"],
        a["kv_rows"], a["batch"], a["n_new"], a["kvh"], a["d"], a["page"], a["ks"], a["vs"],
        a["kind"], a["kss"], a["vss"], a["ndt"], a["kvdt"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("over,status", [
    (dict(kn=None), 1),
    (dict(pos=None), 1),
    (dict(k=None), 1),
    (dict(ws=None), 1),
    (dict(kn=0x1008), 1),                                  # k_new not 16-byte aligned
    (dict(kv_start=None), 1),                              # no layout
    (dict(bt=0x9000, bt_stride=2, page=16), 1),            # both layouts
    (dict(ks=0.0), 1),                                     # 8-bit codes divide by the scale
    (dict(vs=-1.0), 1),
    (dict(ks=float("inf")), 1),
    (dict(ndt=2), 1),                                      # new rows cannot be e4m3
    (dict(ndt=0, kvdt=1), 2),                              # f16 rows into a bf16 cache
    (dict(d=96), 2),
    (dict(kind=2, kvdt=0, kss=0xA000, vss=0xB000), 2),     # finer scales on an f16 cache
    (dict(kind=1), 1),                                     # head scales missing
    (dict(wsb=128), 3),                                    # workspace below the header
    (dict(batch=0), 1),
    (dict(n_new=0), 1),
    (dict(n_new=17), 1),
])
def test_append_host_validation(fda, over, status):
    assert _call_append(fda, **over) == status


def test_decode_with_append_validates_the_append(fda):
    """fd_decode_attention_append refuses a missing new row before any launch."""
    lib = fda.load_library()
    st = lib.fd_decode_attention_append(0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, None, 0,
                                        0x6000, 0x7000, 100, 2, 1, 8, 2, 128, 0, 0.125, 1.0, 1.0,
                                        0, None, None, 0, 2, 0x8000, 0x9000, 0xA000, 1 << 20, None)
    assert st == 1


def test_set_kernel_rejects_unknown(fda):
    lib = fda.load_library()
    assert lib.fd_set_kernel(7) == 1 and lib.fd_set_kernel(5) == 1 and lib.fd_set_kernel(-1) == 1
    for k in (1, 2, 3, 4, 0):
        assert lib.fd_set_kernel(k) == 0


def test_header_enums_match_the_binding(fda):
    """Every enumerator the header defines has the same value in the binding."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(FD_[A-Z0-9_]+)\s*=\s*(\d+)", text))
    for name in ("FD_F16", "FD_BF16", "FD_E4M3", "FD_I8", "FD_SCALE_TENSOR", "FD_SCALE_HEAD",
                 "FD_SCALE_TOKEN", "FD_KERNEL_AUTO", "FD_KERNEL_SIMT", "FD_KERNEL_MMA",
                 "FD_KERNEL_TC", "FD_KERNEL_FMA", "FD_OK",
                 "FD_ERR_INVALID_ARG", "FD_ERR_UNSUPPORTED", "FD_ERR_WORKSPACE_TOO_SMALL",
                 "FD_ERR_CUDA", "FD_ERR_DEVICE_BOUNDS", "FD_ERR_DEVICE_TIMEOUT"):
        assert enums[name] == getattr(fda, name), name


def test_noalloc_classifies_bad_arguments_like_the_workspace_entry(fda):
    """Both entry points give the same status to the same bad arguments
    (checked on the host, before any device work)."""
    lib = fda.load_library()
    fake = 0x1000
    for d, want in ((96, 2), (128, None)):
        st_ws = _call(fda, d=d, qh=8, kvh=2, batch=4)
        st_na = lib.fd_decode_attention_noalloc(fake, fake, fake, fake, None, 0, fake, 100, 4, 8,
                                                2, d, 0, 0.1, 1.0, 1.0, 0, 0, fake, fake, None)
        if want is not None:
            assert st_ws == want and st_na == want, (d, st_ws, st_na)
    for over in (dict(q=None), dict(batch=0), dict(qh=6, kvh=4), dict(kvdt=4)):
        a = dict(q=fake, batch=4, qh=8, kvh=2, kvdt=0)
        a.update(over)
        st_ws = _call(fda, **over)
        st_na = lib.fd_decode_attention_noalloc(a["q"], fake, fake, fake, None, 0, fake, 100,
                                                a["batch"], a["qh"], a["kvh"], 128, 0, 0.1, 1.0,
                                                1.0, 0, a["kvdt"], fake, fake, None)
        assert st_na == st_ws, (over, st_ws, st_na)


def test_debug_hook_arguments_are_checked_on_the_host(fda):
    lib = fda.load_library()
    assert lib.fd_debug_set_wait_limit(-5, 0) == 1
    assert lib.fd_debug_set_wait_limit(0, 0) == 0
    grid = ctypes.c_int(0)
    # no dst, no workspace, bad q_len: refused before any device work
    assert lib.fd_debug_plan_segments(0x1000, None, 2, 1, 8, 2, 128, 0, 0, 0, 0, None, 0, 4,
                                      ctypes.byref(grid), 0x2000, 1 << 20, None) == 1
    assert lib.fd_debug_plan_segments(0x1000, None, 2, 0, 8, 2, 128, 0, 0, 0, 0, 0x3000, 1 << 20,
                                      4, ctypes.byref(grid), 0x2000, 1 << 20, None) == 1
