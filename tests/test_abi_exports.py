"""The C-ABI library loads without a GPU and exports every function include/*.h declares."""
import ctypes
import glob
import os
import re

from prefix_cached_kv_radix_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(api.LIB_PATH)
    names = declared_functions()
    assert {"radix_create", "match_prefix", "insert", "evict", "kv_pool_write", "prefix_extend_attention",
            "decode_attention"} <= names
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(api.EXPORTS) <= names


def test_host_calls_need_no_gpu():
    assert api.version().startswith("radixattn")
    # tracing is off unless asked for; with it on the calls still work (NVTX ranges go nowhere
    # without a profiler) and the setting comes back
    import numpy as np
    assert api.set_tracing(True) is False or os.environ.get("RX_NVTX") == "1"
    t = api.RadixTree(16, 2)
    sl = t.alloc_slots(3)
    t.insert(np.array([5, 6, 7], np.int32), sl)
    assert t.match_prefix_len(np.array([5, 6, 9], np.int32)) == 2
    assert api.set_tracing(False) is True
    t = api.RadixTree(8, 1)
    assert t.stats()["free_slots"] == 8


def test_array_addresses_for_the_binding():
    """The binding's array address helper: the buffer address for writable arrays, the
    array's own for read-only and empty ones (all handed to the library as plain pointers)."""
    import numpy as np
    a = np.arange(10, dtype=np.int32)
    assert api._addr(a) == a.ctypes.data
    ro = np.frombuffer(np.arange(4, dtype=np.int64).tobytes(), np.int64)
    assert not ro.flags.writeable and api._addr(ro) == ro.ctypes.data
    e = np.zeros(0, np.int64)
    assert api._addr(e) == e.ctypes.data
    v = a[2:]                                  # a contiguous view starts where it says
    assert api._addr(v) == a.ctypes.data + 8


def test_step_extension_marshals_like_ctypes():
    """The _rxstep extension writes the step's inputs into the same structs the ctypes path
    writes and returns rx_step_run's code (here RX_EINVAL: no tree, so nothing runs)."""
    import numpy as np
    import pytest
    ext = api.step_ext()
    if ext is None:
        pytest.skip("the Python headers are not installed: the step extension was not built")

    class Dev:   # stands in for a device tensor: only data_ptr() is read
        def __init__(self, p):
            self.p = p

        def data_ptr(self):
            return self.p

    a, io = api.rx_step_args(), api.rx_step_io()
    toks = np.arange(10, dtype=np.int32)
    ind = np.array([0, 4, 10], np.int64)
    nn = np.array([1, 2], np.int32)
    rc = ext.run(ctypes.addressof(a), ctypes.addressof(io), 2, toks, ind, nn, Dev(0x1000), Dev(0x2000), Dev(0x3000),
                 Dev(0x4000), None, 0x5000, 4096)
    assert rc == api.RX_EINVAL
    assert "rx_step_run" in api.load().rx_last_error().decode()
    assert (a.batch, a.tokens, a.tok_indptr, a.n_new) == (2, toks.ctypes.data, ind.ctypes.data, nn.ctypes.data)
    assert (io.d_q, io.d_k_new, io.d_v_new, io.d_out, io.d_lse) == (0x1000, 0x2000, 0x3000, 0x4000, None)
    assert (io.d_stage, io.d_stage_bytes) == (0x5000, 4096)
    with pytest.raises(TypeError):
        ext.run(ctypes.addressof(a), ctypes.addressof(io), 2, toks)
