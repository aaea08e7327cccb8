"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/kda.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def K():
    from linear_attention_mixer_gb300 import build
    build.build()
    import linear_attention_mixer_gb300 as K
    K.lib()
    return K


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(kda_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("kda_config", "kda_state_alloc", "kda_state_free", "kda_state_reset", "kda_state_snapshot",
                 "kda_state_restore", "kda_decode_token", "kda_decode_tokens", "kda_prefill", "kda_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(K):
    names = declared_functions()
    L = K.lib()
    for n in names:
        assert hasattr(L, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (kda_\w+)$", nm, flags=re.M))
    assert set(names) <= exported
    # and the binding wraps exactly those
    assert {s[0] for s in K.SIGNATURES} == set(names)


def test_config_defaults_and_validation(K):
    cfg = K.kda_config(96, 128, K.KDA_BF16)
    assert (cfg.num_heads, cfg.head_dim, cfg.conv_kernel, cfg.chunk_size) == (96, 128, 4, 64)
    assert cfg.gate_lower_bound == -5.0
    assert cfg.l2_eps == pytest.approx(1e-6) and cfg.rms_eps == pytest.approx(1e-6)
    assert cfg.q_scale == pytest.approx(128 ** -0.5)
    for bad in ((0, 128, 1), (96, 64, 1), (96, 128, 7)):
        with pytest.raises(K.KdaError) as ei:
            K.kda_config(*bad)
        assert ei.value.status == K.KDA_ERR_INVALID
        assert K.kda_last_error()


def test_null_and_bad_arguments_rejected_before_the_device(K):
    L = K.lib()
    cfg = K.kda_config(2, 128, K.KDA_F32)
    params = K.kda_layer_params()
    assert L.kda_state_free(None) == K.KDA_OK
    assert L.kda_state_blob_bytes(None, 1) == 0
    assert L.kda_state_max_slots(None) == 0
    assert L.kda_state_reset(None, None, 0, None) == K.KDA_ERR_INVALID
    assert L.kda_state_snapshot(None, None, 0, None, 0, None) == K.KDA_ERR_INVALID
    assert L.kda_state_restore(None, None, 0, None, 0, None) == K.KDA_ERR_INVALID
    code = ctypes.c_int32()
    assert L.kda_state_poll_error(None, ctypes.byref(code)) == K.KDA_ERR_INVALID
    assert L.kda_decode_token(ctypes.byref(cfg), ctypes.byref(params), None, None, 1,
                              *([None] * 7), None) == K.KDA_ERR_INVALID
    assert L.kda_prefill(ctypes.byref(cfg), ctypes.byref(params), None, None, None, None, 1,
                         *([None] * 7), None) == K.KDA_ERR_INVALID
    assert L.kda_decode_tokens(ctypes.byref(cfg), ctypes.byref(params), None, None, 1, 2,
                               *([None] * 7), None) == K.KDA_ERR_INVALID
    out = ctypes.c_void_p()
    assert L.kda_state_alloc(ctypes.byref(cfg), 0, ctypes.byref(out)) == K.KDA_ERR_INVALID
    assert out.value is None
    assert L.kda_state_alloc(None, 1, ctypes.byref(out)) == K.KDA_ERR_INVALID
    bad = K.kda_config_t(2, 128, 4, 0, 32, -5.0, 1e-6, 1e-6, 0.088)  # unsupported chunk size
    assert L.kda_state_alloc(ctypes.byref(bad), 1, ctypes.byref(out)) == K.KDA_ERR_INVALID
    assert "chunk_size" in K.kda_last_error()


def test_blob_header_layout(K):
    assert ctypes.sizeof(K.kda_blob_header) == 64
    assert K.KDA_BLOB_MAGIC == int.from_bytes(b"KDA1", "little")


def test_binding_marshalling_checks(K):
    import torch
    cfg = K.kda_config(2, 128, K.KDA_F32)
    with pytest.raises(TypeError):
        K.kda_layer_params_from(torch.zeros(3, 256, 4), torch.zeros(256), torch.zeros(2), torch.zeros(128))


def test_gate_proj_arguments_rejected_before_the_device(K):
    """kda_gate_proj checks geometry, workspace and alignment on the host; the
    workspace query returns 0 for the same invalid arguments. T = 0 is a no-op."""
    L = K.lib()
    bf = K.kda_config(96, 128, K.KDA_BF16)
    f32 = K.kda_config(96, 128, K.KDA_F32)
    wide = K.kda_config(200, 128, K.KDA_BF16)
    fake = ctypes.c_void_p(1 << 20)  # an aligned address that is never dereferenced
    args = [fake] * 6
    for cfg, hidden, T, why in ((bf, 100, 16, "multiple of 64"), (f32, 100, 16, "multiple of 64"), (bf, 0, 16, "multiple"),
                                (wide, 7168, 16, "num_heads"), (bf, 7168, -1, "T must be")):
        assert L.kda_gate_proj_workspace_bytes(ctypes.byref(cfg), hidden, T) == 0
        assert L.kda_gate_proj(ctypes.byref(cfg), hidden, T, *args, fake, 1 << 30, None) == K.KDA_ERR_INVALID
        assert why in K.kda_last_error()
    assert L.kda_gate_proj(ctypes.byref(bf), 7168, 16, *args, None, 1 << 30, None) == K.KDA_ERR_INVALID
    assert L.kda_gate_proj(ctypes.byref(bf), 7168, 16, *args, ctypes.c_void_p((1 << 20) + 8), 1 << 30,
                           None) == K.KDA_ERR_INVALID
    assert L.kda_gate_proj(ctypes.byref(bf), 7168, 16, None, *args[1:], fake, 1 << 30, None) == K.KDA_ERR_INVALID
    assert L.kda_gate_proj(ctypes.byref(bf), 7168, 16, ctypes.c_void_p((1 << 20) + 2), *args[1:], fake, 1 << 30,
                           None) == K.KDA_ERR_INVALID
    assert "16-byte aligned" in K.kda_last_error()
    assert L.kda_gate_proj(ctypes.byref(bf), 7168, 0, *args, fake, 0, None) == K.KDA_OK
    # the workspace holds the error word and T x (d + 16 ceil(H / 16)) FP32 sums, for either dtype
    for cfg in (bf, f32):
        assert L.kda_gate_proj_workspace_bytes(ctypes.byref(cfg), 7168, 1000) == 256 + 1000 * (128 + 96) * 4


def test_header_is_plain_c_and_a_c_program_links(K, tmp_path):
    """include/kda.h compiles as C99 with warnings as errors, and a C program links against
    libkda.so and calls it (kda_config and an argument check need no GPU)."""
    src = tmp_path / "use_kda.c"
    src.write_text(
        '#include <stdio.h>\n#include "kda.h"\n'
        "int main(void) {\n"
        "    kda_config_t c;\n"
        "    if (kda_config(&c, 96, 128, KDA_BF16) != KDA_OK) return 1;\n"
        "    if (c.num_heads != 96 || c.head_dim != 128 || c.conv_kernel != 4) return 2;\n"
        "    if (kda_config(&c, 96, 64, KDA_BF16) != KDA_ERR_INVALID) return 3;\n"
        "    if (kda_last_error()[0] == 0) return 4;\n"
        "    if (kda_gate_proj_workspace_bytes(&c, 7168, 10) != 256 + 10 * (128 + 96) * 4) return 5;\n"
        "    printf(\"ok\\n\");\n"
        "    return 0;\n"
        "}\n")
    exe = tmp_path / "use_kda"
    libdir = os.path.dirname(K.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lkda", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
