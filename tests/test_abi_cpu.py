"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point include/ar.h declares; host-side argument checks and the launch
plan arithmetic behave as documented."""
import ctypes
import os

import pytest

import tensor_decode_all_gb300 as tda
from tensor_decode_all_gb300 import ar


@pytest.fixture(scope="module")
def lib():
    tda.build()
    return tda.lib()


def test_every_declared_symbol_is_exported(lib):
    names = tda.declared_symbols()
    assert len(names) >= 14, names
    for n in ("ar_create", "ar_allreduce", "ar_allgather", "ar_destroy", "ar_status", "ar_reset",
              "ar_strerror"):
        assert n in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ar.h but not exported"


def test_strerror_names_every_code(lib):
    for code, name in ar.CODE_NAMES.items():
        assert tda.strerror(code).startswith(name)
    assert "unknown" in tda.strerror(999)


def test_create_rejects_bad_arguments_before_touching_cuda(lib):
    for args in [(0, 1, 10, 0), (9, 1, 10, 0), (2, 0, 10, 0), (2, 4, 10, 0), (2, 1, 0, 0), (2, 1, 10, 2),
                 (2, 1, 10, -1)]:
        assert tda.ar_create(*args) == 0
        assert tda.ar_last_error() == ar.AR_EINVAL, args


def test_null_handle_calls(lib):
    assert tda.ar_allreduce(0, 0, 16, 16, 8, 123) == ar.AR_EINVAL
    assert tda.ar_allgather(0, 0, 16, 16, 8, 123) == ar.AR_EINVAL
    assert tda.ar_reset(0) == ar.AR_EINVAL
    assert tda.ar_destroy(0) == ar.AR_OK
    assert tda.ar_set_timeout(0, 10**9) == ar.AR_EINVAL
    assert lib.ar_status(None, None) == ar.AR_EINVAL
    assert lib.ar_query(None, None) == ar.AR_EINVAL


@pytest.mark.parametrize("algo", [ar.AR_ALGO_ONESHOT, ar.AR_ALGO_TWOSHOT, ar.AR_ALGO_TAGGED])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("vec", [16, 8, 2, 1])
def test_plan_invariants(lib, R, vec, algo):
    if algo != ar.AR_ALGO_ONESHOT and vec != 16:
        with pytest.raises(tda.ArError):
            tda.ar_plan_compute(R, 4096, vec, algo, 256, 152, 6)
        return
    sms, bps, threads = 152, 6, 256
    bmax = sms * bps // R
    sizes = [1, 15, 16, 17, 4095, 4096, 8192, 262144, 786432, 1 << 24, (1 << 26) + 12345, 3 << 27]
    for nbytes in sizes:
        if nbytes % vec:
            continue
        p = tda.ar_plan_compute(R, nbytes, vec, algo, threads, sms, bps)
        nv = -(-nbytes // vec)
        assert p.threads == threads and p.vec_bytes == vec and p.algo == algo
        if algo == ar.AR_ALGO_TWOSHOT:
            assert p.flag_rounds == 2 and p.subtile_vecs in (64, 128, 256)
            assert p.tile_bytes == R * p.subtile_vecs * vec          # R sub-tiles per tile
            assert p.unroll == -(-R * p.subtile_vecs // threads)
        else:
            assert p.unroll in (1, 2) and p.flag_rounds == 1
        if algo == ar.AR_ALGO_TAGGED:
            # one 16-byte payload vector per thread per stage (two tagged vectors)
            assert p.unroll == 1 and p.tile_bytes == threads * vec and p.subtile_vecs == 0
        if algo == ar.AR_ALGO_ONESHOT:
            assert p.tile_bytes == threads * p.unroll * vec and p.subtile_vecs == 0
        # tiles cover the payload, and no tile is empty
        tile_vecs = p.tile_bytes // vec
        assert p.tiles * tile_vecs >= nv > (p.tiles - 1) * tile_vecs
        # every block has at least one tile; all ranks' blocks fit at once
        assert 1 <= p.blocks <= min(p.tiles, bmax)
        assert R * p.blocks <= sms * bps
        assert p.max_stages == -(-p.tiles // p.blocks)
        # one-shot, small payloads: one tile per block, spread as wide as allowed
        if algo == ar.AR_ALGO_ONESHOT and nv <= bmax * threads:
            assert p.unroll == 1 and p.max_stages == 1


def test_plan_zero_bytes_and_bad_args(lib):
    p = tda.ar_plan_compute(2, 0, 16, ar.AR_ALGO_ONESHOT, 256, 152, 6)
    assert p.blocks == 0 and p.tiles == 0
    with pytest.raises(tda.ArError):
        tda.ar_plan_compute(9, 16, 16, ar.AR_ALGO_ONESHOT, 256, 152, 6)
    with pytest.raises(tda.ArError):
        tda.ar_plan_compute(2, 16, 3, ar.AR_ALGO_ONESHOT, 256, 152, 6)
    with pytest.raises(tda.ArError):
        tda.ar_plan_compute(2, 16, 16, ar.AR_ALGO_AUTO, 256, 152, 6)  # the caller resolves AUTO
    with pytest.raises(tda.ArError):
        tda.ar_plan_compute(8, 16, 16, ar.AR_ALGO_ONESHOT, 256, 1, 1)  # 8 ranks cannot each get a block


def test_choose_algo_rule(lib):
    for R in (1, 2, 3):
        assert tda.ar_choose_algo(R, 1 << 30, ar.AR_SLOT_HBM) == ar.AR_ALGO_ONESHOT
    for R in (1, 2):
        assert tda.ar_choose_algo(R, 1 << 30, ar.AR_SLOT_PINNED_HOST) == ar.AR_ALGO_ONESHOT
        assert tda.ar_choose_algo(R, 16, ar.AR_SLOT_PINNED_HOST) == ar.AR_ALGO_ONESHOT
    # tagged-word form for small calls (R, HBM limit, pinned limit; 0 = never)
    for R, hbm, pinned in ((1, 512 << 10, 0), (2, 512 << 10, 0), (3, 256 << 10, 0),
                           (4, 64 << 10, 0), (5, 0, 0), (6, 0, 0), (8, 0, 0)):
        for kind, lim in ((ar.AR_SLOT_HBM, hbm), (ar.AR_SLOT_PINNED_HOST, pinned)):
            if lim:
                assert tda.ar_choose_algo(R, 16, kind) == ar.AR_ALGO_TAGGED
                assert tda.ar_choose_algo(R, lim, kind) == ar.AR_ALGO_TAGGED
            assert tda.ar_choose_algo(R, lim + 16, kind) != ar.AR_ALGO_TAGGED
    # thresholds from the measured crossover (R, HBM, pinned host)
    for R, hbm, pinned in ((3, None, 512 << 10), (4, 2 << 20, 128 << 10), (5, 2 << 20, 64 << 10),
                           (7, 2 << 20, 64 << 10), (8, 512 << 10, 32 << 10)):
        if hbm:
            assert tda.ar_choose_algo(R, hbm - 1, ar.AR_SLOT_HBM) == ar.AR_ALGO_ONESHOT
            assert tda.ar_choose_algo(R, hbm, ar.AR_SLOT_HBM) == ar.AR_ALGO_TWOSHOT
        assert tda.ar_choose_algo(R, pinned - 1, ar.AR_SLOT_PINNED_HOST) == ar.AR_ALGO_ONESHOT
        assert tda.ar_choose_algo(R, pinned, ar.AR_SLOT_PINNED_HOST) == ar.AR_ALGO_TWOSHOT
    assert tda.ar_set_algo(0, ar.AR_ALGO_ONESHOT) == ar.AR_EINVAL


def test_struct_layouts_match_header(lib, tmp_path):
    """Every field of the binding's structs sits where a C compiler puts it
    for include/ar.h (sizes and offsets printed by a program built with gcc)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    from tensor_decode_all_gb300 import trace
    structs = {"ar_error_info": ar.ErrorInfo, "ar_info": ar.Info, "ar_plan": ar.Plan, "ar_tactics": ar.Tactics,
               "ar_trace_record": trace.TraceRecord}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "ar.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'    printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-I", os.path.dirname(ar._build.INCLUDE + "/"), str(src), "-o", str(exe)],
                   check=True)
    got = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c = {tuple(l.split()[:2]): int(l.split()[2]) for l in got if l.strip()}
    for cname, py in structs.items():
        assert ctypes.sizeof(py) == c[(cname, "size")], cname
        for fname, _ in py._fields_:
            assert getattr(py, fname).offset == c[(cname, fname)], (cname, fname)


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(ar, "_lib", None)
    monkeypatch.setattr(ar._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        ar.lib()


def test_binding_refuses_tensors_the_pointers_cannot_describe():
    """The Python binding checks what raw pointers hide (dense layout, the
    handle's dtype, room in the output) before any call reaches the library;
    tensors that pass go on to the handle (here a destroyed one)."""
    import torch
    h = ar.Handle.__new__(ar.Handle)
    h.R, h.dtype, h._h = 3, ar.AR_F16, 0
    x = torch.zeros(64, dtype=torch.float16)
    bad = [
        (x[::2], torch.zeros(32, dtype=torch.float16), "not contiguous"),
        (x, torch.zeros(64, dtype=torch.bfloat16), "dtype"),
        (torch.zeros(64, dtype=torch.float32), torch.zeros(64, dtype=torch.float32), "dtype"),
        (x, torch.zeros(63, dtype=torch.float16), "holds 63"),
    ]
    for inp, out, msg in bad:
        with pytest.raises(ValueError, match=msg):
            h.allreduce(0, inp, out)
    with pytest.raises(ValueError, match="holds 64"):
        h.allgather(0, x, torch.zeros(64, dtype=torch.float16))     # needs R * 64
    with pytest.raises(ValueError, match="rank 1's input"):
        h.allreduce_fused([x, x[:32], x], [x, x, x])
    with pytest.raises(ValueError, match="need 3"):
        h.allreduce_fused([x, x], [x, x])
    with pytest.raises(RuntimeError, match="destroyed"):
        h.allreduce(0, x, torch.zeros(64, dtype=torch.float16))
    with pytest.raises(RuntimeError, match="destroyed"):
        h.allgather(0, x, torch.zeros(3 * 64, dtype=torch.float16))


def test_header_is_plain_c_and_cpp(tmp_path):
    """include/ar.h stands alone for a C caller (C99 and C11, pedantic,
    warnings as errors) and a C++ caller (declarations get C linkage)."""
    import shutil
    import subprocess
    inc = os.path.dirname(ar._build.INCLUDE + "/")
    gcc, gxx = shutil.which("gcc"), shutil.which("g++")
    if gcc is None or gxx is None:
        pytest.skip("no C/C++ compiler")
    c = tmp_path / "use.c"
    c.write_text('#include "ar.h"\nint f(void) { ar_tactics t; ar_plan p; (void)t; (void)p; '
                 'return (int)sizeof(ar_error_info) + AR_OK; }\n')
    for std in ("c99", "c11"):
        subprocess.run([gcc, f"-std={std}", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", inc, "-c", str(c),
                        "-o", str(tmp_path / f"use_{std}.o")], check=True)
    cc = tmp_path / "use.cc"
    cc.write_text('#include "ar.h"\n#include "ar.h"\n'
                  'extern "C" int probe() { return ar_last_error(); }\n'
                  'int g() { return (int)sizeof(ar_info) + probe(); }\n')
    obj = tmp_path / "use_cc.o"
    subprocess.run([gxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", inc, "-c", str(cc), "-o", str(obj)],
                   check=True)
    syms = subprocess.run(["nm", str(obj)], check=True, capture_output=True, text=True).stdout
    assert " U ar_last_error" in syms      # an unmangled (C linkage) reference
