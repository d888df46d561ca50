"""CPU-only: the C library's host-side argument checks.  Every call below is rejected
(or, for empty batches, accepted) before any device work, so it runs without a GPU; the
pointers are aligned or misaligned addresses that the library never dereferences on
the host."""
import pytest

OK, INVALID, UNSUPPORTED, NO_BLOCKS, CUDA, WORKSPACE = 0, 1, 2, 3, 4, 5
F16, BF16, FP8 = 0, 1, 2
A = 0x10000          # 16-byte (and 256-byte) aligned fake device address
MIS = 0x10008        # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_187_gb300 import build
    build.build()
    import paged_kv_cache_187_gb300 as pkg
    return pkg.raw()


def _err(lib):
    return (lib.pa_last_error() or b"").decode()


def _v1(lib, **kw):
    p = dict(out=A, q=A, kc=A, vc=A, bt=A, maxb=4, lens=A, S=2, Hq=8, Hkv=2, D=128, bs=16,
             NB=64, mcl=64, scale=0.1, dt=BF16)
    p.update(kw)
    return lib.pa_decode_v1(p["out"], p["q"], p["kc"], p["vc"], p["bt"], p["maxb"], p["lens"],
                            p["S"], p["Hq"], p["Hkv"], p["D"], p["bs"], p["NB"], p["mcl"],
                            p["scale"], p["dt"], None, None)


def _v2(lib, P=64, ws=A, ws_bytes=1 << 30, **kw):
    p = dict(out=A, q=A, kc=A, vc=A, bt=A, maxb=4, lens=A, S=2, Hq=8, Hkv=2, D=128, bs=16,
             NB=64, mcl=64, scale=0.1, dt=BF16)
    p.update(kw)
    return lib.pa_decode_v2(p["out"], p["q"], p["kc"], p["vc"], p["bt"], p["maxb"], p["lens"],
                            p["S"], p["Hq"], p["Hkv"], p["D"], p["bs"], p["NB"], p["mcl"],
                            p["scale"], p["dt"], P, ws, ws_bytes, None, None)


@pytest.mark.parametrize("kw,code,word", [
    (dict(D=96), UNSUPPORTED, "head_size"),
    (dict(bs=8), UNSUPPORTED, "block_size"),
    (dict(dt=FP8), UNSUPPORTED, "dtype"),
    (dict(Hq=12, Hkv=8), INVALID, "num_kv_heads"),
    (dict(Hq=64, Hkv=2), UNSUPPORTED, "group"),
    (dict(S=-1), INVALID, "positive"),
    (dict(Hkv=0), INVALID, "positive"),
    (dict(NB=1 << 27, Hkv=2, bs=16), UNSUPPORTED, "rows"),
    (dict(out=0), INVALID, "null"),
    (dict(lens=0), INVALID, "null"),
    (dict(q=MIS), INVALID, "aligned"),
    (dict(kc=MIS), INVALID, "aligned"),
])
def test_decode_v1_rejects_before_any_launch(lib, kw, code, word):
    assert _v1(lib, **kw) == code
    assert word in _err(lib)


def test_empty_batch_is_a_no_op(lib):
    # no sequences: nothing to launch, even with null buffers
    assert _v1(lib, S=0, out=0, q=0, kc=0, vc=0, bt=0, lens=0) == OK
    assert _v2(lib, S=0, out=0, q=0, kc=0, vc=0, bt=0, lens=0, ws=0, ws_bytes=0) == OK
    assert lib.pa_reshape_and_cache(0, 0, 0, 0, 0, 0, 2, 128, 16, 64, BF16, None, None) == OK


@pytest.mark.parametrize("P,ws,ws_bytes,code,word", [
    (24, A, 1 << 30, INVALID, "partition_size"),     # not a multiple of block_size
    (0, A, 1 << 30, INVALID, "partition_size"),
    (64, 0, 1 << 30, WORKSPACE, "workspace"),
    (64, A, 256, WORKSPACE, "workspace"),
    (64, A + 16, 1 << 30, INVALID, "256-byte"),
])
def test_decode_v2_partition_and_workspace_checks(lib, P, ws, ws_bytes, code, word):
    assert _v2(lib, P=P, ws=ws, ws_bytes=ws_bytes) == code
    assert word in _err(lib)


@pytest.mark.parametrize("args,code,word", [
    (dict(n=-1), INVALID, "positive"),
    (dict(dt=FP8), UNSUPPORTED, "dtype"),
    (dict(D=12), UNSUPPORTED, "multiple of 8"),
    (dict(key=0), INVALID, "null"),
    (dict(key=MIS), INVALID, "aligned"),
])
def test_reshape_and_cache_checks(lib, args, code, word):
    p = dict(key=A, value=A, kc=A, vc=A, slots=A, n=4, Hkv=2, D=128, bs=16, NB=64, dt=BF16)
    p.update(args)
    assert lib.pa_reshape_and_cache(p["key"], p["value"], p["kc"], p["vc"], p["slots"], p["n"],
                                    p["Hkv"], p["D"], p["bs"], p["NB"], p["dt"], None, None) == code
    assert word in _err(lib)


def _fp8(lib, D=128, ks=0.5, vs=0.5, variant=1, **kw):
    return lib.pa_decode_fp8(A, A, A, A, A, 4, A, 2, 8, 2, D, 16, 64, 64, 0.1, ks, vs, BF16,
                             variant, 0, A, 1 << 30, None, None)


@pytest.mark.parametrize("kw,code,word", [
    (dict(D=64), UNSUPPORTED, "head_size 128"),
    (dict(ks=0.0), INVALID, "k_scale"),
    (dict(vs=-1.0), INVALID, "k_scale"),
    (dict(variant=3), INVALID, "variant"),
])
def test_decode_fp8_checks(lib, kw, code, word):
    assert _fp8(lib, **kw) == code
    assert word in _err(lib)


@pytest.mark.parametrize("q_len,Hkv,variant,code,word", [
    (0, 2, 1, INVALID, "q_len"),
    (2, 0, 1, INVALID, "positive"),
    (2, 2, 7, INVALID, "variant"),
    (1 << 18, 2, 1, INVALID, "q_len"),          # q_len * num_q_heads beyond 2^20
])
def test_decode_mq_checks(lib, q_len, Hkv, variant, code, word):
    assert lib.pa_decode_mq(A, A, A, A, A, 4, A, 2, q_len, 8, Hkv, 128, 16, 64, 64, 0.1, BF16,
                            variant, 0, A, 1 << 30, None, None) == code
    assert word in _err(lib)


def _noalloc(lib, P=64, **kw):
    p = dict(out=A, q=A, kc=A, vc=A, bt=A, maxb=4, lens=A, S=2, Hq=8, Hkv=2, D=128, bs=16,
             NB=64, mcl=64, scale=0.1, dt=BF16)
    p.update(kw)
    return lib.pa_decode_v2_noalloc(p["out"], p["q"], p["kc"], p["vc"], p["bt"], p["maxb"],
                                    p["lens"], p["S"], p["Hq"], p["Hkv"], p["D"], p["bs"], p["NB"],
                                    p["mcl"], p["scale"], p["dt"], P, None, None)


def test_noalloc_checks_arguments_before_its_scratch_size(lib):
    huge = 1 << 22
    # valid arguments whose partials exceed the fixed scratch: PA_ERR_WORKSPACE, no launch
    assert _noalloc(lib, P=16, S=64, Hq=32, Hkv=8, mcl=huge, maxb=huge // 16) == WORKSPACE
    assert "scratch" in _err(lib)
    # the same sizes with a bad argument report that argument, as pa_decode_v2 does
    assert _noalloc(lib, P=16, S=64, Hq=32, Hkv=8, D=96, mcl=huge, maxb=huge // 16) == UNSUPPORTED
    assert _v2(lib, P=16, S=64, Hq=32, Hkv=8, D=96, mcl=huge, maxb=huge // 16) == UNSUPPORTED
    assert _noalloc(lib, P=24, mcl=huge, maxb=huge // 16) == INVALID
    assert "partition_size" in _err(lib)
    assert _noalloc(lib, out=MIS) == INVALID


def test_noalloc_scratch_size_agrees_between_header_and_binding():
    import os
    import re
    import paged_kv_cache_187_gb300 as pa
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "pa.h")).read()
    m = re.search(r"#define\s+PA_NOALLOC_SCRATCH_BYTES\s+(.+)", text)
    expr = m.group(1).replace("(size_t)", "")
    assert pa.PA_NOALLOC_SCRATCH_BYTES == eval(expr, {}) == 64 << 20


def test_per_device_set_up_runs_once_per_device_ordinal(tmp_path):
    """The launchers' shared-memory attribute bookkeeping (pa_once.h), compiled into a
    host-only program: set-up runs once on each of two device ordinals, a failed attempt
    is retried, and eight threads racing on both ordinals still run it once per device."""
    import os
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if not gxx:
        pytest.skip("g++ not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "once.cpp"
    src.write_text(r'''
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>
#include "pa_once.h"
int main() {
    pa::PerDeviceOnce once;
    int calls[3] = {0, 0, 0};
    auto set_up = [&](int dev) { return once.run(dev, [&] { ++calls[dev]; return 0; }); };
    if (set_up(0) || set_up(0) || set_up(1) || set_up(1) || set_up(0)) return 1;
    if (calls[0] != 1 || calls[1] != 1 || !once.done(0) || !once.done(1) || once.done(2)) return 2;
    // a failing set-up (e.g. an attribute the device refused) is tried again
    int tries = 0;
    if (once.run(2, [&] { ++tries; return 7; }) != 7 || once.done(2)) return 3;
    if (once.run(2, [&] { ++tries; return 0; }) != 0 || !once.done(2) || tries != 2) return 4;
    // concurrent first calls on two devices
    pa::PerDeviceOnce shared;
    std::atomic<int> per_dev[2];
    per_dev[0] = 0; per_dev[1] = 0;
    std::vector<std::thread> ts;
    for (int t = 0; t < 8; ++t)
        ts.emplace_back([&, t] {
            for (int i = 0; i < 1000; ++i) shared.run((t + i) % 2, [&] { ++per_dev[(t + i) % 2]; return 0; });
        });
    for (auto& th : ts) th.join();
    if (per_dev[0] != 1 || per_dev[1] != 1) return 5;
    std::puts("ok");
    return 0;
}
''')
    exe = tmp_path / "once"
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I",
                    os.path.join(root, "paged_kv_cache_187_gb300", "csrc"), str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
