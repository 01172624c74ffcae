"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/ssd.h, sizes workspaces, and rejects bad arguments on the
host before touching the device."""
import ctypes
import os
import re

import pytest

import mamba_ssd_layer_03_b300 as ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                text = f.read()
            names += re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", text)
    return names


def test_header_declares_entry_points():
    names = _declared_symbols()
    for n in ("ssd_scan", "ssd_scan_workspace_size", "ssd_check_device_status",
              "ssd_status_string", "ssd_resolve_algo"):
        assert n in names


@pytest.mark.parametrize("name", _declared_symbols())
def test_library_exports_declared_symbol(name):
    lib = ssd.load_library()
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_only_declared_symbols_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ssd.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {n for n in exported if n.startswith("ssd_")}
    assert ours == set(_declared_symbols())


def test_status_strings():
    for code in range(7):
        s = ssd.status_string(code)
        assert s.startswith("SSD_")
    assert ssd.status_string(99) == "SSD_ERR_UNKNOWN"


def _shape(**kw):
    import torch
    d = dict(batch=4, seqlen=8192, nheads=80, headdim=64, dstate=128, ngroups=1,
             chunk_size=256, nseq=4, dtype=torch.bfloat16, algo="auto")
    d.update(kw)
    return ssd.make_shape(d["batch"], d["seqlen"], d["nheads"], d["headdim"], d["dstate"],
                          d["ngroups"], d["chunk_size"], d["nseq"], d["dtype"], d["algo"])


def test_workspace_size_simt_scales_with_chunks():
    a = ssd.workspace_size(_shape(algo="simt"))
    b = ssd.workspace_size(_shape(algo="simt", seqlen=16384))
    assert a > 0 and b > a


@pytest.mark.parametrize("kw,code", [
    (dict(chunk_size=100), 2),
    (dict(chunk_size=32), 2),
    (dict(ngroups=3), 1),
    (dict(nheads=0), 1),
    (dict(headdim=300, algo="simt"), 2),
    (dict(dstate=512, algo="simt"), 2),
    (dict(seqlen=-1), 1),
    (dict(seqlen=2**31), 2),
    # buffers that could not exist: rejected before any size is computed from them
    (dict(batch=2**40, seqlen=2**30), 2),
    (dict(batch=2**33, seqlen=2**24, nseq=2**33), 2),
    (dict(batch=1, seqlen=2**24, nheads=2**30, ngroups=1, algo="simt"), 2),          # x: 2^60 elements
    (dict(batch=2**20, seqlen=1, nseq=2**31 - 1, nheads=2**12, dstate=256, algo="simt"), 2),  # states: 2^57
])
def test_workspace_size_rejects(kw, code):
    with pytest.raises(ssd.SsdError) as ei:
        ssd.workspace_size(_shape(**kw))
    assert ei.value.code == code


def test_scan_rejects_on_host_before_device_work():
    lib = ssd.load_library()
    sh = _shape(algo="simt")
    nbytes = ssd.workspace_size(sh)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    args = [fake] * 5 + [None, None, None, fake, None]
    # workspace missing
    assert lib.ssd_scan(ctypes.byref(sh), *args, None, ctypes.c_size_t(0), None) == 3
    # workspace too small
    assert lib.ssd_scan(ctypes.byref(sh), *args, fake, ctypes.c_size_t(nbytes - 1), None) == 3
    # nseq != batch without cu_seqlens
    bad = _shape(algo="simt", nseq=3)
    assert lib.ssd_scan(ctypes.byref(bad), *args, fake, ctypes.c_size_t(nbytes), None) == 1
    # null x with tokens present
    args2 = [None] + [fake] * 4 + [None, None, None, fake, None]
    assert lib.ssd_scan(ctypes.byref(sh), *args2, fake, ctypes.c_size_t(nbytes), None) == 1
    # misaligned bf16 pointer
    odd = ctypes.c_void_p((1 << 20) + 1)
    args3 = [odd] + [fake] * 4 + [None, None, None, fake, None]
    assert lib.ssd_scan(ctypes.byref(sh), *args3, fake, ctypes.c_size_t(nbytes), None) == 2
    # null shape
    assert lib.ssd_scan(None, *args, fake, ctypes.c_size_t(nbytes), None) == 1
    # varlen needs batch == 1
    cu = fake
    args4 = [fake] * 5 + [None, None, cu, fake, None]
    assert lib.ssd_scan(ctypes.byref(sh), *args4, fake, ctypes.c_size_t(nbytes), None) == 1


def test_check_status_rejects_null():
    assert ssd.load_library().ssd_check_device_status(None, None) == 1


# ---------------------------------------------------------------- step-size transform

def test_scan_ex_workspace_with_transform():
    tf = ssd.SsdDtTransform(None, 1, 0.0, float("inf"))
    # the fused kernel applies the transform inline: no extra workspace (its
    # workspace depends on the device's SM count, so this part needs a GPU)
    base = _shape(algo="tc")
    try:
        plain = ssd.workspace_size(base)
    except ssd.SsdError:
        plain = None
    if plain is not None:
        assert ssd.workspace_size(base, tf) == plain
    # the other paths transform dt into the end of the workspace first
    for algo in ("simt", "tc2"):
        sh = _shape(algo=algo)
        try:
            plain = ssd.workspace_size(sh)
        except ssd.SsdError:
            continue   # sized from the device's properties: needs a GPU
        assert ssd.workspace_size(sh, tf) - plain >= 4 * 8192 * 80 * 4, algo


def test_scan_ex_rejects_bad_transform():
    lib = ssd.load_library()
    n = ctypes.c_size_t(0)
    for lo, hi in ((1.0, 0.5), (float("nan"), 1.0)):
        tf = ssd.SsdDtTransform(None, 1, lo, hi)
        assert lib.ssd_scan_ex_workspace_size(ctypes.byref(_shape()), ctypes.byref(tf),
                                              ctypes.byref(n)) == 1


# ---------------------------------------------------------------- decode step

def _step_shape(**kw):
    d = dict(batch=4, nheads=80, headdim=64, dstate=128, ngroups=1, dtype=ssd.SSD_BF16,
             reserved=0)
    d.update(kw)
    return ssd.SsdStepShape(d["batch"], d["nheads"], d["headdim"], d["dstate"], d["ngroups"],
                            d["dtype"], d["reserved"])


@pytest.mark.parametrize("kw,code", [
    (dict(nheads=0), 1),
    (dict(ngroups=3), 1),
    (dict(reserved=1), 1),
    (dict(batch=-1), 1),
    (dict(dtype=7), 2),
    (dict(headdim=2048), 2),
    (dict(dstate=2048), 2),
])
def test_step_rejects_bad_shapes_on_host(kw, code):
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    sh = _step_shape(**kw)
    assert lib.ssd_step(ctypes.byref(sh), fake, fake, None, fake, fake, fake, None, fake, fake,
                        None) == code


def test_step_rejects_null_and_misaligned_pointers():
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)
    sh = _step_shape()
    assert lib.ssd_step(None, fake, fake, None, fake, fake, fake, None, fake, fake, None) == 1
    assert lib.ssd_step(ctypes.byref(sh), None, fake, None, fake, fake, fake, None, fake, fake,
                        None) == 1
    assert lib.ssd_step(ctypes.byref(sh), fake, fake, None, fake, fake, fake, None, None, fake,
                        None) == 1
    odd = ctypes.c_void_p((1 << 20) + 1)
    assert lib.ssd_step(ctypes.byref(sh), odd, fake, None, fake, fake, fake, None, fake, fake,
                        None) == 2
    tf = ssd.SsdDtTransform(None, 1, 2.0, 1.0)
    assert lib.ssd_step(ctypes.byref(sh), fake, fake, ctypes.byref(tf), fake, fake, fake, None,
                        fake, fake, None) == 1


def test_step_zero_batch_is_a_no_op():
    # nothing is enqueued, so null data pointers are fine
    lib = ssd.load_library()
    sh = _step_shape(batch=0)
    assert lib.ssd_step(ctypes.byref(sh), None, None, None, None, None, None, None, None, None,
                        None) == 0


def test_selftest_rejects_bad_arguments():
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.ssd_selftest_wait_timeout(2, fake, None) == 1
    assert lib.ssd_selftest_wait_timeout(0, None, None) == 1


def test_noalloc_rejects_oversized_shape_on_host():
    # checked before the scratch, the device or any pointer is touched
    import ctypes
    lib = ssd.load_library()
    shape = _shape(batch=1, seqlen=2**24, nheads=2**30, ngroups=1, nseq=1, algo="tc")
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.ssd_scan_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake, None, None, fake,
                              None, None, None)
    assert rc == 2, ssd.status_string(rc)


@pytest.mark.parametrize("bad", ["out_shape", "out_dtype", "final_shape", "workspace_dtype"])
def test_scan_checks_caller_buffers_before_any_device_work(bad):
    # meta tensors pass the input checks; a wrong caller-supplied buffer must be
    # refused before the library, the stream or any memory is touched
    import torch
    m = dict(device="meta")
    b, L, H, P, N = 2, 300, 4, 64, 128
    x = torch.empty(b, L, H, P, dtype=torch.bfloat16, **m)
    dt = torch.empty(b, L, H, **m)
    A = torch.empty(H, **m)
    B = torch.empty(b, L, 1, N, dtype=torch.bfloat16, **m)
    kw = dict(out=torch.empty(b, L, H, P, dtype=torch.bfloat16, **m),
              final_out=torch.empty(b, H, P, N, **m))
    if bad == "out_shape":
        kw["out"] = torch.empty(b, L, H, P + 1, dtype=torch.bfloat16, **m)
    elif bad == "out_dtype":
        kw["out"] = torch.empty(b, L, H, P, **m)
    elif bad == "final_shape":
        kw["final_out"] = torch.empty(b, H, P, N // 2, **m)
    else:
        kw["workspace"] = torch.empty(1 << 20, dtype=torch.float32, **m)
    expect = {"out_shape": "out has shape", "out_dtype": "out must be", "final_shape": "final_out has shape",
              "workspace_dtype": "workspace must be"}[bad]
    with pytest.raises((ValueError, TypeError), match=expect):
        ssd.ssd_scan(x, dt, A, B, B, None, 256, algo="simt", **kw)


@pytest.mark.parametrize("field,value", [("chunk_size", 0), ("chunk_size", 64), ("dtype", 0),
                                         ("algo", 1)])
def test_noalloc_rejects_unsupported_shape_before_any_arithmetic(field, value):
    # a chunk size of 0 must come back as UNSUPPORTED, not divide by zero;
    # the allocation-free call takes only what the two-pass kernels take
    import ctypes
    lib = ssd.load_library()
    shape = _shape(batch=1, seqlen=300, nheads=2, ngroups=1, nseq=1, algo="tc")
    setattr(shape, field, value)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the shape check comes first
    rc = lib.ssd_scan_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake, None, None, fake,
                              None, None, None)
    assert rc == 2, ssd.status_string(rc)


@pytest.mark.parametrize("bad", ["dt_shape", "A_dtype", "C_shape", "D_shape", "init_shape",
                                 "x_noncontig", "status_dtype", "algo"])
def test_noalloc_wrapper_checks_inputs_before_the_library(bad):
    # meta tensors: every check runs before the library or any memory is touched
    import torch
    m = dict(device="meta")
    b, L, H, P, N = 2, 300, 4, 64, 128
    a = dict(x=torch.empty(b, L, H, P, dtype=torch.bfloat16, **m), dt=torch.empty(b, L, H, **m),
             A=torch.empty(H, **m), B=torch.empty(b, L, 1, N, dtype=torch.bfloat16, **m),
             C=torch.empty(b, L, 1, N, dtype=torch.bfloat16, **m), D=torch.empty(H, **m))
    kw = {}
    if bad == "dt_shape":
        a["dt"] = torch.empty(b, L, H + 1, **m)
    elif bad == "A_dtype":
        a["A"] = torch.empty(H, dtype=torch.float64, **m)
    elif bad == "C_shape":
        a["C"] = torch.empty(b, L, 1, N // 2, dtype=torch.bfloat16, **m)
    elif bad == "D_shape":
        a["D"] = torch.empty(H + 2, **m)
    elif bad == "init_shape":
        kw["initial_states"] = torch.empty(b, H, P, N + 1, **m)
    elif bad == "x_noncontig":
        a["x"] = torch.empty(b, L, P, H, dtype=torch.bfloat16, **m).transpose(2, 3)
    elif bad == "status_dtype":
        kw["device_status"] = torch.empty(1, dtype=torch.int64, **m)
    else:
        kw["algo"] = "simt"
    with pytest.raises((ValueError, TypeError)):
        ssd.ssd_scan_noalloc(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], 256, **kw)


def test_noalloc_wrapper_refuses_host_tensors():
    import torch
    x = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    B = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        ssd.ssd_scan_noalloc(x, torch.zeros(1, 8, 2), torch.zeros(2), B, B, None, 256)


def test_scan_states_rejects_on_host():
    """ssd_scan_states: shapes the fused kernel does not take, missing
    outputs and short workspaces are refused before any device work."""
    import torch
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced
    ws = ctypes.c_void_p(1 << 24)

    def call(shape, final=fake, wsb=1 << 30, x=fake):
        return lib.ssd_scan_states(ctypes.byref(shape), x, fake, None, fake, fake, None, None,
                                   final, ws, ctypes.c_size_t(wsb), None)

    # (the fused kernel's shapes need the driver's tensor-map encoder, so the
    # checks of those shapes run with the GPU tests)
    assert lib.ssd_scan_states(None, fake, fake, None, fake, fake, None, None, fake, ws,
                               ctypes.c_size_t(1 << 30), None) == 1
    assert call(ssd.make_shape(2, 512, 4, 64, 128, 1, 256, 2, torch.float32, "auto")) == 2
    assert call(ssd.make_shape(2, 512, 4, 32, 128, 1, 256, 2, torch.bfloat16, "auto")) == 2
    assert call(ssd.make_shape(2, 512, 4, 64, 128, 1, 256, 2, torch.bfloat16, "tc2")) == 2
    assert call(ssd.make_shape(2, 512, 4, 64, 128, 1, 256, 2, torch.bfloat16, "simt")) == 2
    assert call(ssd.make_shape(2, 512, 4, 64, 128, 1, 7, 2, torch.bfloat16, "auto")) == 2
