"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from mla_latent_kv_67_b300 import binding as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla_b300.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_path():
    names = declared_functions()
    for want in ("mla_append_latent", "mla_project_q", "mla_absorb_q", "mla_plan_decode",
                 "mla_decode_attn", "mla_combine", "mla_absorb_out", "mla_out_proj",
                 "mla_decode_workspace_size", "mla_rope_table"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = M.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert M.mla_abi_version() == 1


def test_status_strings():
    lib = M.lib()
    assert lib.mla_status_string(0) == b"MLA_OK"
    assert lib.mla_status_string(3) == b"MLA_ERR_WORKSPACE"
    assert lib.mla_status_string(99) == b"MLA_ERR_UNKNOWN"


def _dims(**kw):
    d = dict(n_h=128, d_h=128, d_r=64, d_c=512, d_v=128, d_model=0, d_cq=0, page_size=64)
    d.update(kw)
    return M.Dims(*d.values())


def test_host_validation_rejects_bad_arguments():
    lib = M.lib()
    d = _dims()
    # NULL tensors
    st = lib.mla_absorb_q(None, None, None, 4, M.MLA_BF16, ctypes.byref(d), None)
    assert st == M.MLA_ERR_INVALID_ARG and b"NULL" in lib.mla_last_error()
    # odd RoPE width
    bad = _dims(d_r=63)
    st = lib.mla_absorb_q(None, None, None, 4, M.MLA_BF16, ctypes.byref(bad), None)
    assert st == M.MLA_ERR_INVALID_ARG and b"even" in lib.mla_last_error()
    # unknown dtype
    st = lib.mla_absorb_q(None, None, None, 4, 7, ctypes.byref(d), None)
    assert st == M.MLA_ERR_INVALID_ARG
    # no dims
    st = lib.mla_combine(None, 0, 4, None, None, M.MLA_BF16, None, None)
    assert st == M.MLA_ERR_INVALID_ARG
    # negative batch
    st = lib.mla_decode_attn(None, None, None, 1, 1, None, -1, 1.0, None, 0, None, None,
                             M.MLA_BF16, ctypes.byref(d), None, None)
    assert st == M.MLA_ERR_INVALID_ARG
    # the FP8 staged decode: negative batch, NULL tensors
    st = lib.mla_decode_attn_fp8_staged(None, None, None, 1, 1, None, -1, 1.0, None, 0, None, None,
                                        ctypes.byref(d), None, None)
    assert st == M.MLA_ERR_INVALID_ARG
    st = lib.mla_decode_attn_fp8_staged(None, None, None, 1, 1, None, 2, 1.0, None, 0, None, None,
                                        ctypes.byref(d), None, None)
    assert st == M.MLA_ERR_INVALID_ARG and b"NULL" in lib.mla_last_error()
    assert lib.mla_decode_fp8_staged_workspace_size(0, 4, ctypes.byref(d)) == 0
    assert lib.mla_decode_fp8_staged_workspace_size(2, 0, ctypes.byref(d)) == 0
    # append without d_model
    st = lib.mla_append_latent(1, 1, None, 1, 1, 1, 1, 1, 1, 1, 1, 1, M.MLA_BF16,
                               ctypes.byref(d), None, None)
    assert st == M.MLA_ERR_INVALID_ARG and b"d_model" in lib.mla_last_error()


def test_empty_batch_is_a_no_op():
    lib = M.lib()
    d = _dims()
    assert lib.mla_absorb_q(None, None, None, 0, M.MLA_BF16, ctypes.byref(d), None) == M.MLA_OK
    assert lib.mla_combine(None, 0, 0, None, None, M.MLA_BF16, ctypes.byref(d), None) == M.MLA_OK
    assert lib.mla_decode_attn_fp8_staged(None, None, None, 1, 1, None, 0, 1.0, None, 0, None, None,
                                          ctypes.byref(d), None, None) == M.MLA_OK


def test_binding_refuses_cpu_tensors():
    import torch
    d = _dims(n_h=2, d_h=4, d_r=2, d_c=32, d_v=4)
    q = torch.zeros(1, 2, 6, dtype=torch.bfloat16)
    with pytest.raises(M.MlaError):
        M.mla_absorb_q(q, torch.zeros(8, 32, dtype=torch.bfloat16),
                       torch.zeros(1, 2, 34, dtype=torch.bfloat16), d)


def declared_arity():
    """Parameter count of every function the header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(mla_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    """Every entry the Python binding types has the header's parameter
    count, so a changed C signature cannot silently shift arguments."""
    arity = declared_arity()
    for name, (_, args) in M._SIGS.items():
        assert name in arity, f"{name} is typed in the binding but not declared"
        assert len(args) == arity[name], f"{name}: binding {len(args)} args, header {arity[name]}"


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c(tmp_path, lang, std):
    """The boundary header compiles as strict C99 and as C++ (no CUDA, torch
    or C++-only types in any signature)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip(f"no {lang} compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "mla_b300.h"\nint main(void) { return (int)mla_abi_version(); }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-x", lang,
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_runs_host_calls(tmp_path):
    """A plain C program links against the library and calls it through the
    ABI alone (host-only calls, so no GPU is needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(M.LIB_PATH)
    src = tmp_path / "prog.c"
    src.write_text(
        '#include <stdio.h>\n#include <string.h>\n#include "mla_b300.h"\n'
        'int main(void) {\n'
        '  if (mla_abi_version() != 1) return 1;\n'
        '  if (strcmp(mla_status_string(MLA_OK), "MLA_OK") != 0) return 2;\n'
        '  mla_dims d = {128, 128, 64, 512, 128, 0, 0, 64};\n'
        '  if (mla_absorb_q(NULL, NULL, NULL, 4, MLA_BF16, &d, NULL) != MLA_ERR_INVALID_ARG) return 3;\n'
        '  printf("ok %s\\n", mla_last_error());\n  return 0;\n}\n')
    exe = tmp_path / "prog"
    r = subprocess.run([cc, "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        "-L", libdir, "-lmla_b300", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr)
