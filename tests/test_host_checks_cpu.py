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
