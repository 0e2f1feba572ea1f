"""The C-ABI library loads, exports every entry point its header declares, and
rejects bad arguments on the host before anything is launched.

These run on the CPU: the library is built here by nvcc, and every call below
fails argument checking before any CUDA call. The pointers are fake integers,
so on a machine with a GPU the calls are skipped rather than risk a launch.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
LIB = os.path.join(ROOT, "gated_deltanet_linear_step_gb300", "libgdn.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from gated_deltanet_linear_step_gb300 import _build

        _build.build()
    import gated_deltanet_linear_step_gb300 as g

    return g.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:gdn_status|const char\*|size_t|void|int)\s+(gdn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("gdn_decode_step", "gdn_decode_step_varlen", "gdn_verify_window", "gdn_verify_commit",
               "gdn_decode_step_ex", "gdn_ab_gates", "gdn_in_proj", "gdn_in_proj_workspace_size",
               "gdn_in_proj_noalloc", "gdn_step_inputs", "gdn_proj_pack_bytes", "gdn_pack_proj_weights",
               "gdn_in_proj_packed", "gdn_step_inputs_packed",
               "gdn_last_error", "gdn_get_geometry", "gdn_read_device_error", "gdn_dispatch_kernel"):
        assert fn in names


def test_dispatch_query_refuses_bad_shapes_before_any_cuda_call(lib):
    """gdn_dispatch_kernel checks its shape on the host: a bad one returns -1 with a message and
    never reaches the CUDA runtime (so this runs without a GPU)."""
    import ctypes

    lib.gdn_dispatch_kernel.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gdn_dispatch_kernel.restype = ctypes.c_int
    lib.gdn_last_error.restype = ctypes.c_char_p
    for B, L, T in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1, 1, 100000)]:
        assert lib.gdn_dispatch_kernel(B, L, T) == -1
        assert b"gdn_dispatch_kernel" in lib.gdn_last_error()


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    missing = [fn for fn in declared_functions() if fn not in exported]
    assert not missing, missing
    for fn in declared_functions():
        assert hasattr(lib, fn)


def test_geometry_matches_pages(lib):
    import gated_deltanet_linear_step_gb300 as g

    geo = g.gdn_get_geometry()
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", "geometry.txt")) as f:
        for line in f:
            if not line.startswith("#") and line.strip():
                k, v = line.split()[:2]
                vals[k] = float(v)
    assert geo["head_dim"] == vals["head_dim"]
    assert geo["k_heads"] == vals["k_heads"]
    assert geo["v_heads"] == vals["v_heads"]
    assert geo["conv_channels"] == vals["conv_channels"]
    assert geo["d_conv"] == vals["d_conv"]
    assert geo["value_dim"] == 6144


no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")

B, L, T = 2, 3, 4
SIZES = {  # bytes of each argument of gdn_decode_step for (B, L, T) = (2, 3, 4)
    "qkv": B * L * T * 10240 * 4, "z": B * L * T * 6144 * 4, "alpha": B * L * T * 48 * 4,
    "beta": B * L * T * 48 * 4, "dt": L * 48 * 4, "ssm_a": L * 48 * 4, "conv_w": L * 10240 * 16,
    "ssm_norm": L * 128 * 4, "conv_state": B * L * 10240 * 12, "state": B * L * 48 * 65536, "y": B * L * T * 6144 * 4,
}
ORDER = list(SIZES)


def fake_ptrs():
    """Disjoint, 256-aligned fake addresses for every argument."""
    base, out = 1 << 40, {}
    for k in ORDER:
        out[k] = base
        base += (SIZES[k] + 4095) // 4096 * 4096 + 4096
    return out


def call(lib, p, b=B, l=L, t=T):
    return lib.gdn_decode_step(*[p[k] for k in ORDER], b, l, t, None)


@no_gpu
def test_null_pointer_rejected(lib):
    for k in ORDER:
        p = fake_ptrs()
        p[k] = None
        assert call(lib, p) == 1, k
        assert k in lib.gdn_last_error().decode()


@no_gpu
def test_misaligned_pointer_rejected(lib):
    for k in ORDER:
        p = fake_ptrs()
        p[k] += 4
        assert call(lib, p) == 3, k


@no_gpu
def test_bad_shapes_rejected(lib):
    p = fake_ptrs()
    for b, l, t in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1, 1, 1025), (-1, 2, 2)]:
        assert call(lib, p, b, l, t) == 2, (b, l, t)


@no_gpu
def test_output_aliasing_rejected(lib):
    for out in ("y", "state", "conv_state"):
        for other in ORDER:
            if other == out:
                continue
            p = fake_ptrs()
            p[out] = p[other] + 16 * ((min(SIZES[other], SIZES[out]) // 2) // 16)
            assert call(lib, p) == 4, (out, other)
            assert "overlaps" in lib.gdn_last_error().decode()


@no_gpu
def test_flags_and_window_rules(lib):
    p = fake_ptrs()
    args = [p[k] for k in ORDER]
    assert lib.gdn_decode_step_ex(*args, None, B, L, T, 0x20, None) == 6  # 0x1 to 0x10 are defined
    # the verify window reads the states: y may not overlap them
    w = dict(p)
    w["y"] = w["state"]
    assert lib.gdn_verify_window(*[w[k] for k in ORDER], None, B, L, T, None) == 4
    # the commit needs n_keep
    assert lib.gdn_verify_commit(p["qkv"], p["alpha"], p["beta"], p["dt"], p["ssm_a"], p["conv_w"],
                                 p["conv_state"], p["state"], None, B, L, T, None) == 1
    # misaligned seq_len
    assert lib.gdn_decode_step_varlen(*args, (1 << 39) + 2, B, L, T, None) == 3


@no_gpu
def test_ab_gates_argument_checks(lib):
    base = 1 << 41
    E = 128
    ptr = {"x": base, "wa": base + (1 << 30), "wb": base + (2 << 30), "dt": base + (3 << 30),
           "sa": base + (4 << 30), "gate": base + (5 << 30), "beta": base + (6 << 30)}
    args = lambda p: [p[k] for k in ("x", "wa", "wb", "dt", "sa", "gate", "beta")]  # noqa: E731
    assert lib.gdn_ab_gates(*args(ptr), 2, 3, 1, 100, None) == 2       # n_embd not a multiple of 64
    assert lib.gdn_ab_gates(*args(ptr), 0, 3, 1, E, None) == 2
    p = dict(ptr, wb=None)
    assert lib.gdn_ab_gates(*args(p), 2, 3, 1, E, None) == 1
    p = dict(ptr, gate=ptr["x"] + 64)
    assert lib.gdn_ab_gates(*args(p), 2, 3, 1, E, None) == 4
    p = dict(ptr, beta=ptr["gate"] + 16)
    assert lib.gdn_ab_gates(*args(p), 2, 3, 1, E, None) == 4
    p = dict(ptr, x=ptr["x"] + 8)
    assert lib.gdn_ab_gates(*args(p), 2, 3, 1, E, None) == 3


def test_in_proj_workspace_size(lib):
    # L x token blocks x (n_embd / 64) slices x 2 halves x rows x 128 bytes
    assert lib.gdn_in_proj_workspace_size(64, 36, 1, 2560) == 36 * 1 * 40 * 2 * 64 * 128
    assert lib.gdn_in_proj_workspace_size(1, 1, 1, 64) == 1 * 1 * 1 * 2 * 16 * 128
    assert lib.gdn_in_proj_workspace_size(16, 36, 8, 2560) == 36 * 1 * 40 * 2 * 128 * 128
    assert lib.gdn_in_proj_workspace_size(200, 2, 1, 128) == 2 * 2 * 2 * 2 * 128 * 128
    assert lib.gdn_in_proj_workspace_size(3, 2, 5, 128) == 2 * 1 * 2 * 2 * 16 * 128
    assert lib.gdn_in_proj_workspace_size(0, 2, 5, 128) == 0
    assert lib.gdn_in_proj_workspace_size(2, 2, 5, 100) == 0


@no_gpu
def test_in_proj_argument_checks(lib):
    base = 1 << 41
    E, B, L, T = 128, 2, 3, 1
    ws = lib.gdn_in_proj_workspace_size(B, L, T, E)
    ptr = {"x": base, "wq": base + (1 << 30), "wg": base + (2 << 30), "qkv": base + (3 << 30),
           "z": base + (4 << 30), "ws": base + (5 << 30)}
    args = lambda p: [p[k] for k in ("x", "wq", "wg", "qkv", "z", "ws")]  # noqa: E731
    assert lib.gdn_in_proj(*args(ptr), ws, B, L, T, 100, None) == 2        # n_embd not a multiple of 64
    assert lib.gdn_in_proj(*args(ptr), ws, 0, L, T, E, None) == 2
    assert lib.gdn_in_proj(*args(ptr), ws - 16, B, L, T, E, None) == 2     # workspace too small
    assert lib.gdn_in_proj(*args(dict(ptr, ws=None)), ws, B, L, T, E, None) == 1
    assert lib.gdn_in_proj(*args(dict(ptr, wg=None)), ws, B, L, T, E, None) == 1
    assert lib.gdn_in_proj(*args(dict(ptr, z=ptr["x"] + 64)), ws, B, L, T, E, None) == 4
    assert lib.gdn_in_proj(*args(dict(ptr, z=ptr["qkv"] + 16)), ws, B, L, T, E, None) == 4
    assert lib.gdn_in_proj(*args(dict(ptr, ws=ptr["wq"] + 32)), ws, B, L, T, E, None) == 4
    assert lib.gdn_in_proj(*args(dict(ptr, qkv=ptr["qkv"] + 8)), ws, B, L, T, E, None) == 3


@no_gpu
def test_step_inputs_argument_checks(lib):
    base = 1 << 41
    E, B, L, T = 128, 2, 3, 1
    ws = lib.gdn_in_proj_workspace_size(B, L, T, E)
    keys = ("x", "wq", "wg", "wa", "wb", "dt", "sa", "qkv", "z", "gate", "beta", "ws")
    ptr = {k: base + (i << 32) for i, k in enumerate(keys)}
    args = lambda p: [p[k] for k in keys]  # noqa: E731
    assert lib.gdn_step_inputs(*args(ptr), ws, B, L, T, 100, None) == 2
    assert lib.gdn_step_inputs(*args(ptr), ws - 16, B, L, T, E, None) == 2
    for k in keys:
        assert lib.gdn_step_inputs(*args(dict(ptr, **{k: None})), ws, B, L, T, E, None) == 1, k
        assert lib.gdn_step_inputs(*args(dict(ptr, **{k: ptr[k] + 4})), ws, B, L, T, E, None) == 3, k
    assert lib.gdn_step_inputs(*args(dict(ptr, gate=ptr["beta"] + 16)), ws, B, L, T, E, None) == 4
    assert lib.gdn_step_inputs(*args(dict(ptr, beta=ptr["wa"] + 64)), ws, B, L, T, E, None) == 4
    assert lib.gdn_step_inputs(*args(dict(ptr, ws=ptr["qkv"] + 64)), ws, B, L, T, E, None) == 4


def test_proj_pack_bytes(lib):
    """129 tiles per layer (qkv, gate, alpha/beta) x n_embd / 64 blocks of 16 KB."""
    assert lib.gdn_proj_pack_bytes(36, 2560) == 36 * 129 * 40 * 16384
    assert lib.gdn_proj_pack_bytes(1, 64) == 129 * 16384
    assert lib.gdn_proj_pack_bytes(0, 64) == 0
    assert lib.gdn_proj_pack_bytes(2, 100) == 0
    assert lib.gdn_proj_pack_bytes(2, 65536 + 64) == 0


@no_gpu
def test_pack_and_packed_argument_checks(lib):
    base = 1 << 41
    E, B, L, T = 128, 2, 3, 1
    ws = lib.gdn_in_proj_workspace_size(B, L, T, E)
    pb = lib.gdn_proj_pack_bytes(L, E)
    w = {k: base + (i << 32) for i, k in enumerate(("wq", "wg", "wa", "wb", "pk"))}
    pack = lambda p, n=pb, l=L, e=E: lib.gdn_pack_proj_weights(  # noqa: E731
        p["wq"], p["wg"], p["wa"], p["wb"], p["pk"], n, l, e, None)
    assert pack(dict(w, wq=None)) == 1
    assert pack(dict(w, wa=None)) == 1                  # alpha without beta
    assert lib.gdn_pack_proj_weights(w["wq"], w["wg"], None, None, None, pb, L, E, None) == 1
    assert pack(dict(w, pk=w["pk"] + 8)) == 3
    assert pack(dict(w, wb=w["wb"] + 4)) == 3
    assert pack(w, n=pb - 16) == 2
    assert pack(w, l=0) == 2
    assert pack(w, e=100) == 2
    assert pack(dict(w, pk=w["wg"] + 4096)) == 4        # packed overlaps w_gate
    assert b"overlaps" in lib.gdn_last_error()

    keys = ("x", "pk", "qkv", "z", "ws")
    ptr = {k: base + (i << 32) for i, k in enumerate(keys)}
    proj = lambda p, n=pb, w_=ws, e=E: lib.gdn_in_proj_packed(  # noqa: E731
        p["x"], p["pk"], n, p["qkv"], p["z"], p["ws"], w_, B, L, T, e, None)
    for k in keys:
        assert proj(dict(ptr, **{k: None})) == 1, k
        assert proj(dict(ptr, **{k: ptr[k] + 4})) == 3, k
    assert proj(ptr, n=pb - 16) == 2
    assert proj(ptr, w_=ws - 16) == 2
    assert proj(ptr, e=100) == 2
    assert proj(dict(ptr, qkv=ptr["pk"] + 64)) == 4
    assert proj(dict(ptr, z=ptr["qkv"] + 16)) == 4

    keys = ("x", "pk", "dt", "sa", "qkv", "z", "gate", "beta", "ws")
    ptr = {k: base + (i << 32) for i, k in enumerate(keys)}
    step = lambda p, n=pb: lib.gdn_step_inputs_packed(  # noqa: E731
        p["x"], p["pk"], n, p["dt"], p["sa"], p["qkv"], p["z"], p["gate"], p["beta"], p["ws"], ws, B, L, T, E, None)
    for k in keys:
        assert step(dict(ptr, **{k: None})) == 1, k
        assert step(dict(ptr, **{k: ptr[k] + 4})) == 3, k
    assert step(ptr, n=pb - 16) == 2
    assert step(dict(ptr, gate=ptr["beta"] + 16)) == 4
    assert step(dict(ptr, beta=ptr["pk"] + 64)) == 4


@no_gpu
def test_host_pipeline_argument_checks(lib):
    import ctypes

    base = 1 << 41
    B, L, T = 2, 3, 1
    n = lib.gdn_host_pipeline_slot_bytes(B, L, T)
    assert n > 0 and lib.gdn_host_pipeline_slot_bytes(0, L, T) == 0
    dev = [base + (i << 32) for i in range(6)]  # dt, ssm_a, conv_w, ssm_norm, conv_state, state
    slots = base + (7 << 32)
    h = ctypes.c_void_p()
    assert lib.gdn_host_pipeline_create(None, *dev, None, slots, n, B, L, T, 0) == 1
    assert lib.gdn_host_pipeline_create(ctypes.byref(h), *dev[:5], None, None, slots, n, B, L, T, 0) == 1
    assert lib.gdn_host_pipeline_create(ctypes.byref(h), *dev, None, slots + 16, n, B, L, T, 0) == 3
    assert lib.gdn_host_pipeline_create(ctypes.byref(h), *dev, base + 2, slots, n, B, L, T, 0) == 3
    assert lib.gdn_host_pipeline_create(ctypes.byref(h), *dev, None, slots, n - 256, B, L, T, 0) == 2
    assert lib.gdn_host_pipeline_create(ctypes.byref(h), *dev, None, slots, n, B, L, 0, 0) == 2
    assert b"slots" in lib.gdn_last_error() or b"range" in lib.gdn_last_error()
    assert h.value is None
    assert lib.gdn_host_pipeline_submit(None, base, base, base, base, base) == 1
    assert lib.gdn_host_pipeline_synchronize(None) == 1
    lib.gdn_host_pipeline_destroy(None)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the compiled library every call raises; nothing falls back to another path."""
    import gated_deltanet_linear_step_gb300 as g
    from gated_deltanet_linear_step_gb300 import _binding

    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load_library(str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(_binding.load_library, "__defaults__", (str(tmp_path / "libgdn.so"),))
    t = torch.zeros(1, 1, 1, 10240)
    with pytest.raises(RuntimeError, match="missing"):
        g.gdn_decode_step(t, t, t, t, t, t, t, t, t, t, t)
    with pytest.raises(RuntimeError, match="missing"):
        g.gdn_get_geometry()


def test_oracle_is_not_imported_by_the_product():
    """The library binding and its package never import the oracle."""
    import ast

    pkg = os.path.join(ROOT, "gated_deltanet_linear_step_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            tree = ast.parse(open(os.path.join(pkg, name)).read())
            for node in ast.walk(tree):
                if isinstance(node, ast.Import):
                    assert all(not a.name.startswith("oracle") for a in node.names), name
                elif isinstance(node, ast.ImportFrom):
                    assert not (node.module or "").startswith("oracle"), name
