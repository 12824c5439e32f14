"""ctypes binding of the CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of bench.py, never by the product package.  It shares no code with the
CUDA path; the only thing both sides share is the seeded input generator.

Every function takes numpy arrays on the host.  x and the weights are fp32 arrays, or
uint16 arrays holding bf16 bit patterns (``dtype="bf16"``); all results are fp64 except
integer outputs (int32).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class OracleCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("tau", ctypes.c_double), ("renorm", ctypes.c_int32)]


def load(path=None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        if not _build.up_to_date():
            _build.compile_oracle()
        path = _build.LIB
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    cfgp = ctypes.POINTER(OracleCfg)
    lib.orc_router.argtypes = [cfgp, P, P, P, P, P, P, P]
    lib.orc_dispatch.argtypes = [cfgp, P, P, P, P, P]
    lib.orc_expert.argtypes = [cfgp, P, P, P, P, ctypes.c_int64, ctypes.c_int32, P, P]
    lib.orc_expert_rows.argtypes = [cfgp, P, P, P, P, ctypes.c_int64, P, P, P, P]
    lib.orc_combine.argtypes = [cfgp, P, P, P, P, P, P, P, ctypes.c_int64, P]
    lib.orc_aux.argtypes = [cfgp, P, P, P]
    lib.orc_forward.argtypes = [cfgp] + [P] * 16
    lib.orc_backward.argtypes = [cfgp, P, P, P, P, P, P, P, ctypes.c_double, P, P, P, P, P, P]
    lib.orc_num_threads.argtypes = []
    for f in ("orc_router", "orc_dispatch", "orc_expert", "orc_expert_rows", "orc_combine", "orc_aux",
              "orc_forward", "orc_num_threads", "orc_backward"):
        getattr(lib, f).restype = ctypes.c_int
    if path is None or path == _build.LIB:
        _lib = lib
    return lib


class Oracle:
    """One MoE layer configuration bound to the oracle library.

    ``T, d, E, k, F`` as in the page's notation (tokens, model width, experts, top-k,
    expert hidden width); ``tau`` the router temperature; ``dtype`` "f32" or "bf16" for
    how x and the weights are stored; ``renorm`` renormalises the gates over the k chosen.
    """

    def __init__(self, T, d, E, k, F, tau=1.0, dtype="f32", lib=None, renorm=False):
        self.T, self.d, self.E, self.k, self.F = int(T), int(d), int(E), int(k), int(F)
        self.tau = float(tau)
        self.dtype = dtype
        self.lib = lib if lib is not None else load()
        self.renorm = bool(renorm)
        self.cfg = OracleCfg(self.T, self.d, self.E, self.k, self.F,
                             1 if dtype == "bf16" else 0, self.tau, 1 if renorm else 0)

    # -- helpers -----------------------------------------------------------------
    def _in(self, a):
        if a is None:
            return None
        want = np.uint16 if self.dtype == "bf16" else np.float32
        a = np.ascontiguousarray(a)
        if a.dtype != want:
            raise TypeError(f"expected {want}, got {a.dtype}")
        return a

    @staticmethod
    def _p(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    def _call(self, name, *args):
        rc = getattr(self.lib, name)(ctypes.byref(self.cfg), *args)
        if rc != 0:
            raise RuntimeError(f"{name} failed with code {rc}")

    # -- the method's steps --------------------------------------------------------
    def router(self, x, wr, bias=None):
        """Logits z, softmax p [T,E] (fp64); top-k idx [T,k] int32; gates [T,k] fp64."""
        x, wr = self._in(x), self._in(wr)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        z = np.empty((self.T, self.E), np.float64)
        p = np.empty((self.T, self.E), np.float64)
        idx = np.empty((self.T, self.k), np.int32)
        gate = np.empty((self.T, self.k), np.float64)
        self._call("orc_router", self._p(x), self._p(wr), self._p(b), self._p(z), self._p(p),
                   self._p(idx), self._p(gate))
        return z, p, idx, gate

    def dispatch(self, idx):
        """counts [E], offsets [E+1], perm_src [T k], perm_slot [T k] (all int32)."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        counts = np.empty(self.E, np.int32)
        offsets = np.empty(self.E + 1, np.int32)
        perm_src = np.empty(self.T * self.k, np.int32)
        perm_slot = np.empty(self.T * self.k, np.int32)
        self._call("orc_dispatch", self._p(idx), self._p(counts), self._p(offsets),
                   self._p(perm_src), self._p(perm_slot))
        return counts, offsets, perm_src, perm_slot

    def expert(self, x, w1, w3, w2, t, e):
        """(h [F], out [d]) of expert e applied to token t, fp64."""
        h = np.empty(self.F, np.float64)
        out = np.empty(self.d, np.float64)
        self._call("orc_expert", self._p(self._in(x)), self._p(self._in(w1)),
                   self._p(self._in(w3)), self._p(self._in(w2)), int(t), int(e),
                   self._p(h), self._p(out))
        return h, out

    def expert_rows(self, x, w1, w3, w2, tokens, experts, want_h=True):
        """Row i: (h [F], out [d]) of expert experts[i] on token tokens[i] (fp64), as
        ``expert`` computes one; returns (h [n, F] or None, out [n, d])."""
        tk = np.ascontiguousarray(tokens, dtype=np.int64)
        ex = np.ascontiguousarray(experts, dtype=np.int32)
        if tk.shape != ex.shape or tk.ndim != 1:
            raise ValueError("tokens and experts must be 1-D and of one length")
        n = tk.size
        h = np.empty((n, self.F), np.float64) if want_h else None
        out = np.empty((n, self.d), np.float64)
        self._call("orc_expert_rows", self._p(self._in(x)), self._p(self._in(w1)), self._p(self._in(w3)),
                   self._p(self._in(w2)), n, self._p(tk), self._p(ex), self._p(h), self._p(out))
        return h, out

    def combine(self, x, w1, w3, w2, idx, gate, tokens=None):
        """y rows [len(tokens), d] (fp64) for the given routing; tokens=None -> all."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        if tokens is None:
            tk, n = None, self.T
        else:
            tk = np.ascontiguousarray(tokens, dtype=np.int64)
            n = tk.size
        y = np.empty((n, self.d), np.float64)
        self._call("orc_combine", self._p(self._in(x)), self._p(self._in(w1)),
                   self._p(self._in(w3)), self._p(self._in(w2)), self._p(idx), self._p(gate),
                   self._p(tk), n, self._p(y))
        return y

    def aux(self, p, counts):
        p = np.ascontiguousarray(p, dtype=np.float64)
        counts = np.ascontiguousarray(counts, dtype=np.int32)
        out = ctypes.c_double(0.0)
        self._call("orc_aux", self._p(p), self._p(counts), ctypes.byref(out))
        return out.value

    def forward(self, x, wr, bias, w1, w3, w2):
        """The whole forward: dict with y, idx, gate, counts, offsets, perm_src,
        perm_slot, z, p, aux."""
        T, E, k, d = self.T, self.E, self.k, self.d
        r = dict(y=np.empty((T, d), np.float64), idx=np.empty((T, k), np.int32),
                 gate=np.empty((T, k), np.float64), counts=np.empty(E, np.int32),
                 offsets=np.empty(E + 1, np.int32), perm_src=np.empty(T * k, np.int32),
                 perm_slot=np.empty(T * k, np.int32), z=np.empty((T, E), np.float64),
                 p=np.empty((T, E), np.float64))
        aux = ctypes.c_double(0.0)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self._call("orc_forward", self._p(self._in(x)), self._p(self._in(wr)), self._p(b),
                   self._p(self._in(w1)), self._p(self._in(w3)), self._p(self._in(w2)),
                   self._p(r["y"]), self._p(r["idx"]), self._p(r["gate"]),
                   self._p(r["counts"]), self._p(r["offsets"]), self._p(r["perm_src"]),
                   self._p(r["perm_slot"]), self._p(r["z"]), self._p(r["p"]),
                   ctypes.byref(aux))
        r["aux"] = aux.value
        return r


    def backward(self, x, wr, bias, w1, w3, w2, dy, alpha=0.0):
        """Gradients of L = sum(dy * y) + alpha * aux: dict dx [T,d], dwr [E,d], dbias [E],
        dw1, dw3 [E,F,d], dw2 [E,d,F] (fp64)."""
        T, E, d, F = self.T, self.E, self.d, self.F
        r = dict(dx=np.empty((T, d)), dwr=np.empty((E, d)), dbias=np.empty(E), dw1=np.empty((E, F, d)),
                 dw3=np.empty((E, F, d)), dw2=np.empty((E, d, F)))
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        self._call("orc_backward", self._p(self._in(x)), self._p(self._in(wr)), self._p(b),
                   self._p(self._in(w1)), self._p(self._in(w3)), self._p(self._in(w2)), self._p(dy),
                   float(alpha), self._p(r["dx"]), self._p(r["dwr"]), self._p(r["dbias"]),
                   self._p(r["dw1"]), self._p(r["dw3"]), self._p(r["dw2"]))
        return r


def num_threads():
    return load().orc_num_threads()
