"""GB300 (sm_103a) linear-recurrence state update behind a C ABI.

``scan_runtime_gb300`` is the Python face of ``libsn.so``:

* ``scan_runtime_gb300._abi`` -- the C functions under their C names
  (``sn_scan_fma``, ``sn_recur_rwkv7``, ...), argument marshalling only;
* ``Context`` -- a small convenience wrapper that owns an ``SnCtx``,
  allocates output tensors with PyTorch and raises ``SnError`` on a non-zero
  status.

PyTorch supplies device memory and streams; every step of the recurrences
runs in libsn's kernels.  Nothing here computes a result on the CPU.
"""
from __future__ import annotations

from . import _abi
from ._abi import *  # noqa: F401,F403  (C names and constants)


def build(force: bool = False) -> str:
    """Compile libsn.so for sm_103a (in-tree)."""
    from ._build import build as _b
    return _b(force=force)


class SnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status} ({_abi.sn_status_str(status)})")


def _check(status: int, what: str) -> None:
    if status != _abi.SN_OK:
        raise SnError(status, what)


class Context:
    """Owns an ``SnCtx`` bound to one CUDA device."""

    def __init__(self, device: int = 0):
        import torch
        self.device = device
        self._torch = torch
        s, h = _abi.sn_ctx_create(device)
        _check(s, "sn_ctx_create")
        self.handle = h
        self._ws = None

    def close(self) -> None:
        if getattr(self, "handle", None):
            _abi.sn_ctx_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- ctx
    def set_option(self, key: int, value: int) -> None:
        _check(_abi.sn_ctx_set_option(self.handle, key, value), "sn_ctx_set_option")

    def get_option(self, key: int) -> int:
        s, v = _abi.sn_ctx_get_option(self.handle, key)
        _check(s, "sn_ctx_get_option")
        return v

    def last_error(self) -> int:
        return _abi.sn_ctx_last_error(self.handle)

    def ensure_workspace(self, B: int, T: int, N: int) -> None:
        """Give the context enough workspace for the look-back scan of (B, T, N)."""
        need = _abi.sn_workspace_bytes(_abi.SN_OP_SCAN_FMA, B, T, N)
        if self._ws is not None and self._ws.numel() >= need:
            return
        self._ws = self._torch.empty(max(need, 256), dtype=self._torch.uint8, device=f"cuda:{self.device}")
        _check(_abi.sn_ctx_set_workspace(self.handle, self._ws, self._ws.numel()), "sn_ctx_set_workspace")

    def ensure_workspace_bytes(self, need: int) -> None:
        """Give the context a workspace of at least `need` bytes."""
        if self._ws is not None and self._ws.numel() >= need:
            return
        self._ws = self._torch.empty(max(need, 256), dtype=self._torch.uint8, device=f"cuda:{self.device}")
        _check(_abi.sn_ctx_set_workspace(self.handle, self._ws, self._ws.numel()), "sn_ctx_set_workspace")

    def _out(self, shape, want):
        if want is None or want is False:
            return None
        if want is True:
            return self._torch.empty(shape, dtype=self._torch.float32, device=f"cuda:{self.device}")
        return want

    # ---------------------------------------------------------------- tier 1
    def scan_fma(self, a, b, s0=None, *, s_out=True, s_final=True, stream=None):
        B, T, N = a.shape
        so, sf = self._out((B, T, N), s_out), self._out((B, N), s_final)
        _check(_abi.sn_scan_fma(self.handle, B, T, N, a, b, s0, sf, so, stream), "sn_scan_fma")
        return so, sf

    def scan_gated(self, a, u, s0=None, *, s_out=True, s_final=True, stream=None):
        B, T, N = a.shape
        so, sf = self._out((B, T, N), s_out), self._out((B, N), s_final)
        _check(_abi.sn_scan_gated(self.handle, B, T, N, a, u, s0, sf, so, stream), "sn_scan_gated")
        return so, sf

    def scan_host(self, a, b=None, u=None, s0=None, *, out=None, rows_per_chunk=1):
        """Scan host (CPU, ideally pinned) tensors through the GPU with
        ``sn_scan_host``: the FMA form when ``b`` is given, the gated form when
        ``u`` is given, sharing the upload of ``a``; batch rows stream through
        the device in chunks of ``rows_per_chunk`` on the context's three
        pipeline streams.  Returns ``{"fma": (s_out, s_final), "gated": (...)}``
        as CPU tensors, filled once the call returns; pass ``out`` (the same
        dict shape, pinned tensors) to reuse buffers across calls."""
        torch = self._torch
        B, T, N = a.shape
        forms = [f for f, x in (("fma", b), ("gated", u)) if x is not None]
        if not forms:
            raise ValueError("give b (FMA form), u (gated form) or both")
        outs = dict(out or {})
        for f in forms:
            if f not in outs:
                outs[f] = (torch.empty((B, T, N), pin_memory=True), torch.empty((B, N), pin_memory=True))
        mask = (1 if b is not None else 0) | (2 if u is not None else 0)
        need = _abi.sn_scan_host_staging_bytes(B, T, N, mask, rows_per_chunk)
        if need < 0:
            raise ValueError("invalid dimensions for sn_scan_host")
        if getattr(self, "_staging", None) is None or self._staging.numel() < need:
            self._staging = torch.empty(max(need, 256), dtype=torch.uint8, device=f"cuda:{self.device}")
        fo, go = outs.get("fma", (None, None)), outs.get("gated", (None, None))
        stream = torch.cuda.current_stream(torch.device(f"cuda:{self.device}"))
        _check(_abi.sn_scan_host(self.handle, B, T, N, rows_per_chunk, a, b, u, s0, fo[0], fo[1], go[0], go[1],
                                 self._staging, self._staging.numel(), stream), "sn_scan_host")
        stream.synchronize()
        return outs

    def scan_backward(self, form, a, s, grad_s, *, s0=None, grad_final=None, u=None, stream=None):
        """Reverse scan of `form` ("fma" or "gated"); returns (grad_a, grad_b|grad_u, grad_s0)."""
        B, T, N = a.shape
        ga, gb, g0 = self._out((B, T, N), True), self._out((B, T, N), True), self._out((B, N), True)
        if form == "fma":
            st = _abi.sn_scan_fma_backward(self.handle, B, T, N, a, s0, s, grad_s, grad_final, ga, gb, g0, stream)
        else:
            st = _abi.sn_scan_gated_backward(self.handle, B, T, N, a, u, s0, s, grad_s, grad_final, ga, gb, g0,
                                             stream)
        _check(st, f"sn_scan_{form}_backward")
        return ga, gb, g0

    # ---------------------------------------------------------------- tier 2
    def recur_diag(self, q, k, v, d, S_in=None, *, H, G, decay_kind, scale, S_out=True, o=True, stream=None):
        B, T, _, dk = k.shape
        dv = v.shape[3]
        So, oo = self._out((B, H, dk, dv), S_out), self._out((B, T, H, dv), o)
        _check(_abi.sn_recur_diag(self.handle, B, T, H, G, dk, dv, decay_kind, scale, q, k, v, d, S_in, So, oo,
                                  stream), "sn_recur_diag")
        return oo, So

    def recur_diag_chunked(self, q, k, v, d, S_in=None, *, H, G, decay_kind, scale, S_out=True, o=True,
                           stream=None):
        """Chunked tensor-core form of recur_diag (tf32 operands); sizes the
        context workspace on first use."""
        B, T, _, dk = k.shape
        dv = v.shape[3]
        need = _abi.sn_recur_chunked_workspace_bytes(B, T, H, dk, dv)
        if need < 0:
            raise SnError(_abi.SN_E_INVAL, "sn_recur_chunked_workspace_bytes")
        self.ensure_workspace_bytes(need)
        So, oo = self._out((B, H, dk, dv), S_out), self._out((B, T, H, dv), o)
        _check(_abi.sn_recur_diag_chunked(self.handle, B, T, H, G, dk, dv, decay_kind, scale, q, k, v, d, S_in, So,
                                          oo, stream), "sn_recur_diag_chunked")
        return oo, So

    def readout_norm_gate(self, o, g, w=None, *, eps, y=True, stream=None):
        """GLA readout epilogue y = RMSNorm(o) * w * silu(g); o, g (B, T, H, dv).
        Pass y=o to write in place."""
        B, T, H, dv = o.shape
        yy = self._out((B, T, H, dv), y)
        _check(_abi.sn_readout_norm_gate(self.handle, B, T, H, dv, o, g, w, eps, yy, stream), "sn_readout_norm_gate")
        return yy

    def readout_dskip(self, o, x, D, *, y=True, stream=None):
        """Mamba-2 skip connection y = o + D_h x; o, x (B, T, H, dv), D (H,)."""
        B, T, H, dv = o.shape
        yy = self._out((B, T, H, dv), y)
        _check(_abi.sn_readout_dskip(self.handle, B, T, H, dv, o, x, D, yy, stream), "sn_readout_dskip")
        return yy

    def recur_delta_chunked(self, q, k, v, beta, S_in=None, *, scale, S_out=True, o=True, stream=None):
        """Chunked tensor-core form of recur_delta (tf32 operands); sizes the
        context workspace on first use."""
        B, T, H, dk = k.shape
        dv = v.shape[3]
        need = _abi.sn_recur_delta_chunked_workspace_bytes(B, T, H, dk, dv)
        if need < 0:
            raise SnError(_abi.SN_E_INVAL, "sn_recur_delta_chunked_workspace_bytes")
        self.ensure_workspace_bytes(need)
        So, oo = self._out((B, H, dk, dv), S_out), self._out((B, T, H, dv), o)
        _check(_abi.sn_recur_delta_chunked(self.handle, B, T, H, dk, dv, scale, q, k, v, beta, S_in, So, oo, stream),
               "sn_recur_delta_chunked")
        return oo, So

    def recur_delta(self, q, k, v, beta, S_in=None, *, scale, S_out=True, o=True, stream=None):
        B, T, H, dk = k.shape
        dv = v.shape[3]
        So, oo = self._out((B, H, dk, dv), S_out), self._out((B, T, H, dv), o)
        _check(_abi.sn_recur_delta(self.handle, B, T, H, dk, dv, scale, q, k, v, beta, S_in, So, oo, stream),
               "sn_recur_delta")
        return oo, So

    def recur_rwkv7(self, q, k, v, w, S_in=None, *, S_out=True, o=True, stream=None):
        B, T, H, dk = k.shape
        dv = v.shape[3]
        So, oo = self._out((B, H, dv, dk), S_out), self._out((B, T, H, dv), o)
        _check(_abi.sn_recur_rwkv7(self.handle, B, T, H, dk, dv, q, k, v, w, S_in, So, oo, stream),
               "sn_recur_rwkv7")
        return oo, So
