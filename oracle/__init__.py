"""The fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg import this
package. It wraps ``oracle.c`` (plain C, fp64, OpenMP) through ctypes and shares no code with
the CUDA library. Every function is pinned by the CPU tests; see the header of ``oracle.c``
for the pages and sections each one follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

CONTIGUOUS, ZIGZAG, STRIPED = 0, 1, 2
FULL, DIAG, SKIP = 0, 1, 2
RING, ALLGATHER, ULYSSES = 0, 1, 2

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def compile_source(src: str, out: str) -> str:
    """Compile one C file of the oracle into a shared library (also used by the mutation tests)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(SOURCE):
        return _OUT
    return compile_source(SOURCE, _OUT)


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_token_of.argtypes = [_I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64]
    lib.oracle_token_of.restype = _I64
    lib.oracle_layout_map.argtypes = [_I64, ctypes.c_int, ctypes.c_int, _P]
    lib.oracle_chunk_assignment.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.oracle_attention.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P,
                                     ctypes.c_int, ctypes.c_double, _I64, _P, _I64, _P, _P, _P]
    lib.oracle_ring.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P,
                                ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P]
    lib.oracle_merge.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
    lib.oracle_merge.restype = None
    lib.oracle_classify.argtypes = [_I64, _P, _I64, _P, ctypes.c_int]
    lib.oracle_plan_counts.argtypes = [_I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int,
                                       ctypes.c_int, _P, _P, _P, _P]
    lib.oracle_half_units.argtypes = [_I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.oracle_cp_comm_bytes.argtypes = [ctypes.c_double] * 4 + [ctypes.c_int]
    lib.oracle_cp_comm_bytes.restype = ctypes.c_double
    lib.oracle_ulysses_breakeven.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.oracle_ulysses_breakeven.restype = ctypes.c_double
    lib.oracle_overlap_min_tokens.argtypes = [ctypes.c_double] * 4
    lib.oracle_overlap_min_tokens.restype = ctypes.c_double
    lib.oracle_kv_bytes_recv.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_kv_bytes_recv.restype = _I64
    lib.oracle_attention_docs.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                          _P, _P, ctypes.c_int, ctypes.c_double, _I64, _P, _P, _P]
    lib.oracle_attention_backward.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                              _P, _P, ctypes.c_int, ctypes.c_double, _I64, _P, _I64, _P, _P, _P, _P]
    lib.oracle_attention_backward_docs.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P,
                                                   _P, _P, _P, _P, ctypes.c_int, ctypes.c_double, _I64, _P, _I64, _P,
                                                   _P, _P, _P]
    lib.oracle_ring_backward.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P,
                                         _P, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _P, _P, _P]
    lib.oracle_bwd_bytes_recv.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_bwd_bytes_recv.restype = _I64
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


class Oracle:
    """Python face of one compiled oracle library (the committed one, or a test's mutant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else _load()

    # -- placement ---------------------------------------------------------------------
    def token_of(self, T, n_cp, layout, r, j) -> int:
        return int(self.lib.oracle_token_of(T, n_cp, layout, r, j))

    def layout_map(self, T, n_cp, layout) -> np.ndarray:
        out = np.empty(T, dtype=np.int64)
        if self.lib.oracle_layout_map(T, n_cp, layout, out.ctypes.data):
            raise ValueError("bad layout arguments")
        return out.reshape(n_cp, T // n_cp)

    def chunk_assignment(self, n_cp, layout, r):
        buf = (ctypes.c_int * 2)()
        k = self.lib.oracle_chunk_assignment(n_cp, layout, r, buf)
        return [buf[i] for i in range(k)]

    # -- attention ---------------------------------------------------------------------
    def attention(self, q, k, v, causal=True, scale=None, pos=None, rows=None, keys=None):
        """q [B,T,h,d], k/v [B,T,n_kv,d] as uint16 bf16 bits. Returns (o [B,R,h,d], lse [B,h,R]) fp64.

        rows: natural token ids of the queries (default all); keys: natural token ids the
        queries may attend to (default all), still subject to the causal mask."""
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        rowsp, R = None, T
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            rowsp, R = rows.ctypes.data, rows.size
        keysp, K = None, T
        if keys is not None:
            keys = np.ascontiguousarray(keys, dtype=np.int64)
            keysp, K = keys.ctypes.data, keys.size
        o = np.empty((B, R, h, d), dtype=np.float64)
        lse = np.empty((B, h, R), dtype=np.float64)
        rc = self.lib.oracle_attention(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data, posp,
                                       int(causal), scale, R, rowsp, K, keysp, o.ctypes.data, lse.ctypes.data)
        if rc:
            raise ValueError("oracle_attention failed")
        return o, lse

    def attention_docs(self, q, k, v, doc, causal=True, scale=None, pos=None, rows=None):
        """attention() under a document mask: doc [T] int document id per natural token."""
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        doc = np.ascontiguousarray(doc, dtype=np.int32)
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        rowsp, R = None, T
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            rowsp, R = rows.ctypes.data, rows.size
        o = np.empty((B, R, h, d), dtype=np.float64)
        lse = np.empty((B, h, R), dtype=np.float64)
        rc = self.lib.oracle_attention_docs(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data, posp,
                                            doc.ctypes.data, int(causal), scale, R, rowsp, o.ctypes.data,
                                            lse.ctypes.data)
        if rc:
            raise ValueError("oracle_attention_docs failed")
        return o, lse

    def ring(self, q, k, v, n_cp, layout, causal=True, scale=None, pos=None, block=16):
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        o = np.empty((B, T, h, d), dtype=np.float64)
        lse = np.empty((B, h, T), dtype=np.float64)
        rc = self.lib.oracle_ring(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data, posp, int(causal),
                                  scale, n_cp, layout, block, o.ctypes.data, lse.ctypes.data)
        if rc:
            raise ValueError("oracle_ring failed")
        return o, lse

    # -- gradients ----------------------------------------------------------------------
    def backward(self, q, k, v, dout, causal=True, scale=None, pos=None, rows=None, keys=None, doc=None):
        """Gradients of L = sum(O * dO) for bf16-bit inputs (dout [B,T,h,d] bf16 bits too).

        Returns (dq [B,R,h,d] for the query rows `rows`, dk [B,K,n_kv,d], dv [B,K,n_kv,d] for the
        keys `keys`), fp64; rows/keys default to all T. doc: document id per token (document mask)."""
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, dout))
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        rowsp, R = None, T
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            rowsp, R = rows.ctypes.data, rows.size
        keysp, K = None, T
        if keys is not None:
            keys = np.ascontiguousarray(keys, dtype=np.int64)
            keysp, K = keys.ctypes.data, keys.size
        dq = np.empty((B, R, h, d), dtype=np.float64)
        dk = np.empty((B, K, n_kv, d), dtype=np.float64)
        dv = np.empty((B, K, n_kv, d), dtype=np.float64)
        if doc is not None:
            doc = np.ascontiguousarray(doc, dtype=np.int32)
            rc = self.lib.oracle_attention_backward_docs(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                                         dout.ctypes.data, posp, doc.ctypes.data, int(causal), scale, R,
                                                         rowsp, K, keysp, dq.ctypes.data, dk.ctypes.data,
                                                         dv.ctypes.data)
        else:
            rc = self.lib.oracle_attention_backward(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                                    dout.ctypes.data, posp, int(causal), scale, R, rowsp, K, keysp,
                                                    dq.ctypes.data, dk.ctypes.data, dv.ctypes.data)
        if rc:
            raise ValueError("oracle_attention_backward failed")
        return dq, dk, dv

    def ring_backward(self, q, k, v, dout, n_cp, layout, causal=True, scale=None, pos=None, block=16):
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, dout))
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        dq = np.empty((B, T, h, d), dtype=np.float64)
        dk = np.empty((B, T, n_kv, d), dtype=np.float64)
        dv = np.empty((B, T, n_kv, d), dtype=np.float64)
        rc = self.lib.oracle_ring_backward(B, T, h, n_kv, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                           dout.ctypes.data, posp, int(causal), scale, n_cp, layout, block,
                                           dq.ctypes.data, dk.ctypes.data, dv.ctypes.data)
        if rc:
            raise ValueError("oracle_ring_backward failed")
        return dq, dk, dv

    def bwd_bytes_recv(self, B, n, n_kv, d_k, n_cp, grad_bytes) -> int:
        return int(self.lib.oracle_bwd_bytes_recv(B, n, n_kv, d_k, n_cp, grad_bytes))

    def merge(self, o_parts, lse_parts):
        """o_parts [S,rows,h,d], lse_parts [S,h,rows] (fp64). Returns (o [rows,h,d], lse [h,rows])."""
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
        S, rows, h, d = o_parts.shape
        o = np.empty((rows, h, d), dtype=np.float64)
        lse = np.empty((h, rows), dtype=np.float64)
        self.lib.oracle_merge(S, rows, h, d, o_parts.ctypes.data, lse_parts.ctypes.data, o.ctypes.data, lse.ctypes.data)
        return o, lse

    # -- classes, work and bytes -------------------------------------------------------
    def classify(self, qpos, kpos, causal=True) -> int:
        qpos = np.ascontiguousarray(qpos, dtype=np.int64)
        kpos = np.ascontiguousarray(kpos, dtype=np.int64)
        return int(self.lib.oracle_classify(qpos.size, qpos.ctypes.data, kpos.size, kpos.ctypes.data, int(causal)))

    def plan_counts(self, T, n_cp, layout, causal=True, bq=128, bk=128, pos=None):
        full = np.zeros((n_cp, n_cp), dtype=np.int64)
        diag = np.zeros_like(full)
        skip = np.zeros_like(full)
        pairs = np.zeros(n_cp, dtype=np.int64)
        posp = None
        if pos is not None:
            pos = np.ascontiguousarray(pos, dtype=np.int32)
            posp = pos.ctypes.data
        if self.lib.oracle_plan_counts(T, n_cp, layout, int(causal), posp, bq, bk, full.ctypes.data,
                                       diag.ctypes.data, skip.ctypes.data, pairs.ctypes.data):
            raise ValueError("oracle_plan_counts failed")
        return {"full": full, "diag": diag, "skip": skip, "pairs": pairs}

    def half_units(self, T, n_cp, layout, causal=True) -> np.ndarray:
        out = np.zeros(n_cp, dtype=np.int64)
        if self.lib.oracle_half_units(T, n_cp, layout, int(causal), out.ctypes.data):
            raise ValueError("oracle_half_units failed")
        return out

    def cp_comm_bytes(self, T, d, d_kv, n_cp, method) -> float:
        return float(self.lib.oracle_cp_comm_bytes(T, d, d_kv, n_cp, method))

    def ulysses_breakeven(self, h, n_kv) -> float:
        return float(self.lib.oracle_ulysses_breakeven(h, n_kv))

    def overlap_min_tokens(self, flops_per_s, bytes_per_s, h, n_kv) -> float:
        return float(self.lib.oracle_overlap_min_tokens(flops_per_s, bytes_per_s, h, n_kv))

    def kv_bytes_recv(self, B, n, n_kv, d_k, n_cp) -> int:
        return int(self.lib.oracle_kv_bytes_recv(B, n, n_kv, d_k, n_cp))


    # -- Ulysses, the head split ([CEX] "Ulysses, splitting by heads instead") ------------------
    @staticmethod
    def ulysses_heads(h, n_kv, n_cp, r):
        """Query heads and KV heads rank r holds after the first all-to-all: h / n_cp whole query
        heads, and the KV heads those use under the GQA map i -> i // (h / n_kv)."""
        hp = h // n_cp
        heads = list(range(r * hp, (r + 1) * hp))
        g = h // n_kv
        return heads, sorted({i // g for i in heads})

    def ulysses(self, q, k, v, n_cp, causal=True, scale=None, pos=None):
        """The head split run literally: rank r holds tokens r n .. r n + n - 1 (n = T / n_cp) of
        every head; the first all-to-all gives each rank all T tokens of its heads; each rank runs
        the attention definition on them; the second all-to-all returns every rank's outputs to
        the token split. Data movement only around attention(); returns (o [B,T,h,d], lse [B,h,T])."""
        B, T, h, d = q.shape
        n_kv = k.shape[2]
        if h % n_cp or T % n_cp:
            raise ValueError("Ulysses needs whole heads and equal token shards per rank")
        n = T // n_cp
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        shard = [(q[:, r * n:(r + 1) * n], k[:, r * n:(r + 1) * n], v[:, r * n:(r + 1) * n]) for r in range(n_cp)]
        o_shard = [np.empty((B, n, h, d)) for _ in range(n_cp)]
        lse_shard = [np.empty((B, h, n)) for _ in range(n_cp)]
        for rr in range(n_cp):
            heads, kvh = self.ulysses_heads(h, n_kv, n_cp, rr)
            # the rank's local GQA map must be the global one: local head i uses local KV head
            # i // (len(heads) / len(kvh)) in attention()
            g_loc = len(heads) // len(kvh)
            assert all(heads[i] // (h // n_kv) == kvh[i // g_loc] for i in range(len(heads)))
            qh = np.concatenate([shard[r][0][:, :, heads] for r in range(n_cp)], axis=1)
            kh = np.concatenate([shard[r][1][:, :, kvh] for r in range(n_cp)], axis=1)
            vh = np.concatenate([shard[r][2][:, :, kvh] for r in range(n_cp)], axis=1)
            o_r, lse_r = self.attention(qh, kh, vh, causal=causal, scale=scale, pos=pos)
            for r in range(n_cp):                        # second all-to-all
                o_shard[r][:, :, heads] = o_r[:, r * n:(r + 1) * n]
                lse_shard[r][:, heads] = lse_r[:, :, r * n:(r + 1) * n]
        return np.concatenate(o_shard, axis=1), np.concatenate(lse_shard, axis=2)

    def ulysses_bytes_recv(self, B, T, h, n_kv, d_k, n_cp) -> np.ndarray:
        """Bytes each rank receives in the two all-to-alls of one forward pass, counted rank pair
        by rank pair: from every other rank, its n tokens of the receiver's query heads and KV
        heads (K and V), and back, the receiver's own n tokens of the sender's output heads;
        2 bytes a number."""
        n = T // n_cp
        out = np.zeros(n_cp, dtype=np.int64)
        for r in range(n_cp):
            heads, kvh = self.ulysses_heads(h, n_kv, n_cp, r)
            for src in range(n_cp):
                if src == r:
                    continue
                src_heads, _ = self.ulysses_heads(h, n_kv, n_cp, src)
                numbers = n * d_k * (len(heads) + 2 * len(kvh)) + n * d_k * len(src_heads)
                out[r] += 2 * B * numbers
        return out

_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
