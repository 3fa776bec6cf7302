"""The C-ABI library loads and exports every entry point include/lookahead.h declares (CPU only)."""
import ctypes as C
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    src = open(os.path.join(ROOT, "include", "lookahead.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from lookahead_decoding_gb300 import build
    build()
    from lookahead_decoding_gb300 import _lib
    names = declared()
    assert "la_init" in names and "la_step" in names and "la_generate" in names
    missing = [n for n in names if not hasattr(_lib.LIB, n)]
    assert missing == []
    assert set(names) <= set(_lib.EXPORTS)


def test_argument_errors_need_no_gpu():
    from lookahead_decoding_gb300 import _lib
    L = _lib.LIB
    assert L.la_strerror(0) == b"ok" and L.la_strerror(3) == b"call out of order"
    out = C.c_void_p()
    # null pointers and bad shapes are rejected before any CUDA call
    assert L.la_init(None, None, 64, 5, 3, 5, None, C.byref(out)) == _lib.LA_EINVAL
    cfg = _lib.la_model_cfg(2, 128, 4, 4, 32, 512, 512, 1e-5, 1e4, 0)
    w = _lib.la_weights()
    assert L.la_init(C.byref(cfg), C.byref(w), 64, 5, 3, 5, None, C.byref(out)) == _lib.LA_EINVAL   # null weights
    bad = _lib.la_model_cfg(2, 100, 4, 4, 32, 512, 512, 1e-5, 1e4, 0)                                # d != H*dh
    assert L.la_init(C.byref(bad), C.byref(w), 64, 5, 3, 5, None, C.byref(out)) == _lib.LA_EINVAL
    nd = _lib.la_model_cfg(2, 128, 4, 4, 32, 512, 512, 1e-5, 1e4, 7)                                 # unknown dtype
    assert L.la_init(C.byref(nd), C.byref(w), 64, 5, 3, 5, None, C.byref(out)) == _lib.LA_ENOTSUP
    assert L.la_step(None, 5, 3, 5, None, None, None) == _lib.LA_EINVAL
    assert L.la_generate(None, None, 0, 1, 5, 3, 5, None, None, None, None) == _lib.LA_EINVAL
    assert L.la_free(None) is None


def test_generate_batch_marshalling(monkeypatch):
    """The binding passes the prompts back to back with their lengths and
    cuts the B x max_new output into one list per request (a recording
    stand-in replaces the library call; no GPU)."""
    from lookahead_decoding_gb300 import _lib
    seen = {}

    class Stub:
        def la_generate_batch(self, ctx, B, flat, lengths, max_new, W, N, G, sampling, out, stats):
            seen.update(B=B, flat=[flat[i] for i in range(9)], lengths=[lengths[i] for i in range(B)],
                        knobs=(max_new, W, N, G))
            for b in range(B):
                for i in range(max_new):
                    out[b * max_new + i] = 100 * b + i
            return 0

    monkeypatch.setattr(_lib, "LIB", Stub())
    got = _lib.la_generate_batch(None, [[1, 2], [3, 4, 5, 6], [7, 8, 9]], 3, 5, 4, 2)
    assert seen == {"B": 3, "flat": [1, 2, 3, 4, 5, 6, 7, 8, 9], "lengths": [2, 4, 3], "knobs": (3, 5, 4, 2)}
    assert got == [[0, 1, 2], [100, 101, 102], [200, 201, 202]]
