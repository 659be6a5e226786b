"""GB300-native DSpark draft/verify hot path.

Python binding of the C ABI declared in ``include/dsd.h``.  This module only
marshals arguments (device pointers of torch tensors, the current CUDA
stream) into ``libdsd.so``; every step of the path runs in the library's
CUDA kernels.  If the library is not built, or no sm_100-family GPU is
present, the calls fail loudly: there is no CPU fallback.

Low-level functions carry the C names (``dsd_propose`` ...).  ``Context``
wraps them with output allocation for convenience.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdsd.so")

DSD_OK = 0
STATUS_NAMES = {
    0: "DSD_OK", -1: "DSD_ERR_ARG", -2: "DSD_ERR_ALIGN", -3: "DSD_ERR_DTYPE",
    -4: "DSD_ERR_SHAPE", -5: "DSD_ERR_CUDA", -6: "DSD_ERR_NONFINITE",
    -7: "DSD_ERR_TIMEOUT", -8: "DSD_ERR_CAPACITY", -9: "DSD_ERR_UNSUPPORTED",
}
DTYPES = {"f32": 0, "bf16": 1}
TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}
ACTS = {"none": 0, "silu": 1}
ENGINES = {"auto": 0, "simt": 1, "tcgen05": 2, "mma": 3}

EXPORTED = [
    "dsd_create", "dsd_destroy", "dsd_last_error", "dsd_sync_status", "dsd_workspace_bytes",
    "dsd_launch_count", "dsd_last_engine", "dsd_last_p_in_place",
    "dsd_propose", "dsd_schedule", "dsd_verify", "dsd_cycle", "dsd_cycle_host", "dsd_overlap",
    "dsd_propose_noalloc", "dsd_loss_forward", "dsd_confidence_head", "dsd_threshold_keep",
    "dsd_calibration", "dsd_propose_gated", "dsd_verify_gated", "dsd_propose_candidates",
    "dsd_propose_rnn", "dsd_verify_rnn", "dsd_gumbel_noise", "dsd_wait_selftest",
    "dsd_auroc", "dsd_auroc_scratch_bytes",
]


class DsdError(RuntimeError):
    def __init__(self, code, msg=""):
        self.code = code
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")


class dsd_config(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int), ("rank", ctypes.c_int), ("gamma", ctypes.c_int),
                ("R_max", ctypes.c_int), ("dtype", ctypes.c_int), ("act", ctypes.c_int),
                ("bias_at_first", ctypes.c_int), ("engine", ctypes.c_int),
                ("device", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_U64 = ctypes.c_uint64


def load_library(path: str | None = None):
    """Load libdsd.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    sig = {
        "dsd_create": (_I, [ctypes.POINTER(dsd_config), ctypes.POINTER(_P)]),
        "dsd_destroy": (_I, [_P]),
        "dsd_last_error": (ctypes.c_char_p, [_P]),
        "dsd_sync_status": (_I, [_P, _P]),
        "dsd_workspace_bytes": (ctypes.c_size_t, [_P]),
        "dsd_launch_count": (_U64, [_P]),
        "dsd_last_engine": (_I, [_P]),
        "dsd_last_p_in_place": (_I, [_P]),
        "dsd_propose": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _F, _U64, _P, _P, _P, _P, _P]),
        "dsd_schedule": (_I, [_P, _I, _P, _P, _I, _P, _P, _P]),
        "dsd_verify": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _U64, _P, _P, _P]),
        "dsd_cycle": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _F, _U64,
                           _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "dsd_cycle_host": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _F, _U64,
                                _P, _P, _P, _P, _P]),
        "dsd_overlap": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "dsd_loss_forward": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _P, _P,
                                  _P]),
        "dsd_propose_candidates": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _F, _U64, _P, _P, _P, _P,
                                        _P, _P, _P]),
        "dsd_propose_gated": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _F, _U64, _P, _P,
                                   _P, _P, _P, _P]),
        "dsd_verify_gated": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _U64,
                                  _P, _P, _P]),
        "dsd_gumbel_noise": (_I, [_P, _P, _I, _P]),
        "dsd_wait_selftest": (_I, [_P, ctypes.c_uint32, _P, _P]),
        "dsd_auroc_scratch_bytes": (ctypes.c_size_t, [_I, _I]),
        "dsd_auroc": (_I, [_P, _I, _P, _P, _P, ctypes.c_size_t, _P, _P]),
        "dsd_propose_rnn": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _F, _U64, _P, _P,
                                 _P, _P, _P, _P]),
        "dsd_verify_rnn": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _U64,
                                _P, _P, _P]),
        "dsd_confidence_head": (_I, [_P, _I, _I, _P, _P, _P, _F, _P, _P, _P, _P, _P]),
        "dsd_threshold_keep": (_I, [_P, _I, _P, _F, _P, _P]),
        "dsd_calibration": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P]),
        "dsd_propose_noalloc": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _F,
                                     _U64, _P, _P, _P, _P, _P, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x):
    """Device/host pointer of a tensor, an int address, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    return int(x)


def _stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(ctx, rc):
    if rc != DSD_OK:
        msg = load_library().dsd_last_error(ctx).decode(errors="replace") if ctx else ""
        raise DsdError(rc, msg)


# ------------------------------------------------------------ C-named calls

def dsd_create(V, rank, gamma, R_max, dtype="bf16", act="none", bias_at_first=True,
               engine="auto", device=0):
    lib = load_library()
    cfg = dsd_config(V, rank, gamma, R_max, DTYPES[dtype], ACTS[act], int(bool(bias_at_first)),
                     ENGINES[engine], device)
    out = _P()
    rc = lib.dsd_create(ctypes.byref(cfg), ctypes.byref(out))
    if rc != DSD_OK:
        raise DsdError(rc, "dsd_create")
    return out


def dsd_destroy(ctx):
    return load_library().dsd_destroy(ctx)


def dsd_sync_status(ctx, stream=None, device=0):
    return load_library().dsd_sync_status(ctx, _stream(stream, device))


def dsd_propose(ctx, R, U, E, W, conf, prev_tok, req_id, temperature, seed, tokens, lse_q,
                logit_at_tok, survival, stream=None, device=0):
    _check(ctx, load_library().dsd_propose(
        ctx, R, _ptr(U), _ptr(E), _ptr(W), _ptr(conf), _ptr(prev_tok), _ptr(req_id),
        float(temperature), int(seed) & (2 ** 64 - 1), _ptr(tokens), _ptr(lse_q),
        _ptr(logit_at_tok), _ptr(survival), _stream(stream, device)))


def dsd_schedule(ctx, R, survival, sps, n_sps, keep_len, theta_B, stream=None, device=0):
    _check(ctx, load_library().dsd_schedule(
        ctx, R, _ptr(survival), _ptr(sps), int(n_sps), _ptr(keep_len), _ptr(theta_B),
        _stream(stream, device)))


def dsd_verify(ctx, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len, req_id,
               temperature, seed, accept_len, next_token, stream=None, device=0):
    _check(ctx, load_library().dsd_verify(
        ctx, R, _ptr(P), _ptr(U), _ptr(E), _ptr(W), _ptr(prev_tok), _ptr(tokens), _ptr(lse_q),
        _ptr(logit_at_tok), _ptr(keep_len), _ptr(req_id), float(temperature),
        int(seed) & (2 ** 64 - 1), _ptr(accept_len), _ptr(next_token), _stream(stream, device)))


def dsd_cycle(ctx, R, U, E, W, conf, prev_tok, req_id, P, sps, n_sps, temperature, seed, tokens,
              lse_q, logit_at_tok, survival, keep_len, theta_B, accept_len, next_token,
              stream=None, device=0):
    _check(ctx, load_library().dsd_cycle(
        ctx, R, _ptr(U), _ptr(E), _ptr(W), _ptr(conf), _ptr(prev_tok), _ptr(req_id), _ptr(P),
        _ptr(sps), int(n_sps), float(temperature), int(seed) & (2 ** 64 - 1), _ptr(tokens),
        _ptr(lse_q), _ptr(logit_at_tok), _ptr(survival), _ptr(keep_len), _ptr(theta_B),
        _ptr(accept_len), _ptr(next_token), _stream(stream, device)))


def dsd_cycle_host(ctx, R, U_host, E, W, conf_host, prev_tok_host, req_id_host, P_host, sps,
                   n_sps, temperature, seed, tokens_host, keep_len_host, accept_len_host,
                   next_token_host, stream=None, device=0):
    _check(ctx, load_library().dsd_cycle_host(
        ctx, R, _ptr(U_host), _ptr(E), _ptr(W), _ptr(conf_host), _ptr(prev_tok_host),
        _ptr(req_id_host), _ptr(P_host), _ptr(sps), int(n_sps), float(temperature),
        int(seed) & (2 ** 64 - 1), _ptr(tokens_host), _ptr(keep_len_host),
        _ptr(accept_len_host), _ptr(next_token_host), _stream(stream, device)))


def dsd_overlap(ctx, N, P_logits, Q_logits, valid_len, a, l1, tau, accept_rate, mean_tau,
                stream=None, device=0):
    _check(ctx, load_library().dsd_overlap(
        ctx, N, _ptr(P_logits), _ptr(Q_logits), _ptr(valid_len), _ptr(a), _ptr(l1), _ptr(tau),
        _ptr(accept_rate), _ptr(mean_tau), _stream(stream, device)))


def dsd_loss_forward(ctx, B, U, E, W, prev_tok, P, target, conf_logit, ce_alpha, l1_alpha,
                     conf_alpha, decay, row_out, losses, stream=None, device=0):
    _check(ctx, load_library().dsd_loss_forward(
        ctx, B, _ptr(U), _ptr(E), _ptr(W), _ptr(prev_tok), _ptr(P), _ptr(target),
        _ptr(conf_logit), ce_alpha, l1_alpha, conf_alpha, decay, _ptr(row_out), _ptr(losses),
        _stream(stream, device)))


def dsd_propose_candidates(ctx, R, U, E, W, conf, prev_tok, req_id, temperature, seed, tokens,
                           lse_q, logit_at_tok, survival, cand_tok, cand_logit, stream=None,
                           device=0):
    _check(ctx, load_library().dsd_propose_candidates(
        ctx, R, _ptr(U), _ptr(E), _ptr(W), _ptr(conf), _ptr(prev_tok), _ptr(req_id), temperature,
        seed, _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok), _ptr(survival), _ptr(cand_tok),
        _ptr(cand_logit), _stream(stream, device)))


def dsd_propose_gated(ctx, R, U, E, W, h, H, W_g, conf, prev_tok, req_id, temperature, seed,
                      tokens, lse_q, logit_at_tok, survival, gated_rep, stream=None, device=0):
    _check(ctx, load_library().dsd_propose_gated(
        ctx, R, _ptr(U), _ptr(E), _ptr(W), _ptr(h), H, _ptr(W_g), _ptr(conf), _ptr(prev_tok),
        _ptr(req_id), temperature, seed, _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok),
        _ptr(survival), _ptr(gated_rep), _stream(stream, device)))


def dsd_verify_gated(ctx, R, P, U, E, W, gated_rep, prev_tok, tokens, lse_q, logit_at_tok,
                     keep_len, req_id, temperature, seed, accept_len, next_token, stream=None,
                     device=0):
    _check(ctx, load_library().dsd_verify_gated(
        ctx, R, _ptr(P), _ptr(U), _ptr(E), _ptr(W), _ptr(gated_rep), _ptr(prev_tok),
        _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok), _ptr(keep_len), _ptr(req_id), temperature,
        seed, _ptr(accept_len), _ptr(next_token), _stream(stream, device)))


def dsd_gumbel_noise(words, out, stream=None, device=0):
    """out[i] = the Gumbel noise of Philox word words[i] (int32 / uint32 bits,
    device tensors), as the sampled kernels draw it."""
    rc = load_library().dsd_gumbel_noise(_ptr(words), _ptr(out), int(words.numel()),
                                         _stream(stream, device))
    if rc != 0:
        raise DsdError(rc, "dsd_gumbel_noise")
    return out


def dsd_propose_rnn(ctx, R, U, E, W, h, H, W_rnn, conf, prev_tok, req_id, temperature, seed,
                    tokens, lse_q, logit_at_tok, survival, rnn_rep, stream=None, device=0):
    _check(ctx, load_library().dsd_propose_rnn(
        ctx, R, _ptr(U), _ptr(E), _ptr(W), _ptr(h), H, _ptr(W_rnn), _ptr(conf), _ptr(prev_tok),
        _ptr(req_id), temperature, seed, _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok),
        _ptr(survival), _ptr(rnn_rep), _stream(stream, device)))


def dsd_verify_rnn(ctx, R, P, U, E, W, rnn_rep, prev_tok, tokens, lse_q, logit_at_tok,
                   keep_len, req_id, temperature, seed, accept_len, next_token, stream=None,
                   device=0):
    _check(ctx, load_library().dsd_verify_rnn(
        ctx, R, _ptr(P), _ptr(U), _ptr(E), _ptr(W), _ptr(rnn_rep), _ptr(prev_tok),
        _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok), _ptr(keep_len), _ptr(req_id), temperature,
        seed, _ptr(accept_len), _ptr(next_token), _stream(stream, device)))


def dsd_confidence_head(ctx, R, H, h, E, w_c, b_c, prev_tok, tokens, conf, survival,
                        stream=None, device=0):
    _check(ctx, load_library().dsd_confidence_head(
        ctx, R, H, _ptr(h), _ptr(E), _ptr(w_c), b_c, _ptr(prev_tok), _ptr(tokens), _ptr(conf),
        _ptr(survival), _stream(stream, device)))


def dsd_threshold_keep(ctx, R, conf, threshold, keep_len, stream=None, device=0):
    _check(ctx, load_library().dsd_threshold_keep(ctx, R, _ptr(conf), threshold, _ptr(keep_len),
                                                  _stream(stream, device)))


def dsd_calibration(ctx, M, conf, accept_len, n_bins, bins, pos, metrics, stream=None, device=0):
    _check(ctx, load_library().dsd_calibration(ctx, M, _ptr(conf), _ptr(accept_len), n_bins,
                                               _ptr(bins), _ptr(pos), _ptr(metrics),
                                               _stream(stream, device)))


def dsd_auroc_scratch_bytes(M, gamma):
    return int(load_library().dsd_auroc_scratch_bytes(int(M), int(gamma)))


def dsd_auroc(ctx, M, conf, accept_len, scratch, auroc, stream=None, device=0):
    """AUROC of predicted survival against realised survival, into the device
    double `auroc`; `scratch` is a caller-owned uint8 device tensor of at least
    dsd_auroc_scratch_bytes(M, gamma) bytes."""
    nbytes = scratch.numel() * scratch.element_size() if isinstance(scratch, torch.Tensor) else 0
    _check(ctx, load_library().dsd_auroc(ctx, int(M), _ptr(conf), _ptr(accept_len), _ptr(scratch),
                                         nbytes, _ptr(auroc), _stream(stream, device)))


def dsd_wait_selftest(ctx, poll_limit, roles_out=None, stream=None, device=0):
    """Run the bounded-wait self-test kernel (a wait that never completes
    must end in DSD_ERR_TIMEOUT, read by dsd_sync_status)."""
    _check(ctx, load_library().dsd_wait_selftest(ctx, int(poll_limit), _ptr(roles_out),
                                                 _stream(stream, device)))


def dsd_propose_noalloc(V, rank, gamma, dtype, act, bias_at_first, R, U, E, W, conf, prev_tok,
                        req_id, temperature, seed, tokens, lse_q, logit_at_tok, survival,
                        status=None, stream=None, device=0):
    """Propose without a context and without allocating device memory (for
    callers that may not allocate); scratch lives in a fixed array inside the
    library.  R * gamma <= 1024.  ``status`` (optional int32 device tensor of
    one element) receives the call's device-side status."""
    rc = load_library().dsd_propose_noalloc(
        int(V), int(rank), int(gamma), DTYPES[dtype] if isinstance(dtype, str) else int(dtype),
        ACTS[act] if isinstance(act, str) else int(act), int(bool(bias_at_first)), int(R),
        _ptr(U), _ptr(E), _ptr(W), _ptr(conf), _ptr(prev_tok), _ptr(req_id), float(temperature),
        int(seed) & (2 ** 64 - 1), _ptr(tokens), _ptr(lse_q), _ptr(logit_at_tok), _ptr(survival),
        _ptr(status), _stream(stream, device))
    if rc != DSD_OK:
        raise DsdError(rc, "dsd_propose_noalloc")


# ------------------------------------------------------------ convenience

class Context:
    """One library context bound to one GPU.  Allocates outputs with torch;
    all computation happens in libdsd.so."""

    def __init__(self, V, rank, gamma, R_max, dtype="bf16", act="none", bias_at_first=True,
                 engine="auto", device=0):
        if not torch.cuda.is_available():
            raise RuntimeError("no CUDA device: the DSpark hot path has no CPU fallback")
        self.V, self.rank, self.gamma, self.R_max = V, rank, gamma, R_max
        self.dtype, self.device = dtype, device
        self.torch_dtype = TORCH_DTYPES[dtype]
        self._dev = torch.device("cuda", device)
        self.handle = dsd_create(V, rank, gamma, R_max, dtype, act, bias_at_first, engine, device)

    def close(self):
        if self.handle:
            dsd_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def workspace_bytes(self):
        return load_library().dsd_workspace_bytes(self.handle)

    def launch_count(self):
        return int(load_library().dsd_launch_count(self.handle))

    def last_engine(self):
        """'simt' or 'tcgen05': the engine of the last propose call."""
        code = int(load_library().dsd_last_engine(self.handle))
        return {v: k for k, v in ENGINES.items()}.get(code, "auto")

    def last_p_in_place(self):
        """True if the last cycle_host call read P in place from host memory."""
        return bool(load_library().dsd_last_p_in_place(self.handle))

    def sync_status(self, stream=None):
        return dsd_sync_status(self.handle, stream, self.device)

    def _empty(self, shape, dtype):
        return torch.empty(shape, dtype=dtype, device=self._dev)

    def _check_in(self, name, t, dtype=None):
        if t is None:
            return
        if not isinstance(t, torch.Tensor) or t.device != self._dev:
            raise ValueError(f"{name} must be a tensor on {self._dev}")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")

    def propose(self, U, E, W, conf, prev_tok, req_id=None, temperature=0.0, seed=0,
                out=None, stream=None):
        R = U.shape[0]
        for n, t in (("U", U), ("E", E), ("W", W)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("conf", conf, torch.float32)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("req_id", req_id, torch.int32)
        G = self.gamma
        o = out or dict(tokens=self._empty((R, G), torch.int32),
                        lse_q=self._empty((R, G), torch.float32),
                        logit_at_tok=self._empty((R, G), torch.float32),
                        survival=self._empty((R, G), torch.float32))
        dsd_propose(self.handle, R, U, E, W, conf, prev_tok, req_id, temperature, seed,
                    o["tokens"], o["lse_q"], o["logit_at_tok"], o["survival"], stream, self.device)
        return o

    def propose_candidates(self, U, E, W, conf, prev_tok, req_id=None, temperature=0.0, seed=0,
                           out=None, stream=None):
        """dsd_propose plus the Markov top-16 candidate set of every position:
        cand_tok [R, gamma, 16] i32 and cand_logit [R, gamma, 16] f32."""
        R = U.shape[0]
        for n, t in (("U", U), ("E", E), ("W", W)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("conf", conf, torch.float32)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("req_id", req_id, torch.int32)
        G = self.gamma
        o = out or dict(tokens=self._empty((R, G), torch.int32),
                        lse_q=self._empty((R, G), torch.float32),
                        logit_at_tok=self._empty((R, G), torch.float32),
                        survival=self._empty((R, G), torch.float32),
                        cand_tok=self._empty((R, G, 16), torch.int32),
                        cand_logit=self._empty((R, G, 16), torch.float32))
        dsd_propose_candidates(self.handle, R, U, E, W, conf, prev_tok, req_id, temperature, seed,
                               o["tokens"], o["lse_q"], o["logit_at_tok"], o["survival"],
                               o["cand_tok"], o["cand_logit"], stream, self.device)
        return o

    def propose_gated(self, U, E, W, h, W_g, conf, prev_tok, req_id=None, temperature=0.0,
                      seed=0, out=None, stream=None):
        """dsd_propose with the gated Markov head; h [R, gamma, H], W_g
        [rank, H + rank].  Also returns gated_rep [R, gamma, rank] f32."""
        R, G, H = h.shape
        for n, t in (("U", U), ("E", E), ("W", W), ("h", h), ("W_g", W_g)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("conf", conf, torch.float32)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("req_id", req_id, torch.int32)
        o = out or dict(tokens=self._empty((R, G), torch.int32),
                        lse_q=self._empty((R, G), torch.float32),
                        logit_at_tok=self._empty((R, G), torch.float32),
                        survival=self._empty((R, G), torch.float32),
                        gated_rep=self._empty((R, G, self.rank), torch.float32))
        dsd_propose_gated(self.handle, R, U, E, W, h, H, W_g, conf, prev_tok, req_id, temperature,
                          seed, o["tokens"], o["lse_q"], o["logit_at_tok"], o["survival"],
                          o["gated_rep"], stream, self.device)
        return o

    def verify_gated(self, P, tokens, keep_len, gated_rep=None, U=None, E=None, W=None,
                     prev_tok=None, lse_q=None, logit_at_tok=None, req_id=None, temperature=0.0,
                     seed=0, out=None, stream=None):
        R = P.shape[0]
        self._check_in("P", P, self.torch_dtype)
        self._check_in("tokens", tokens, torch.int32)
        self._check_in("keep_len", keep_len, torch.int32)
        self._check_in("gated_rep", gated_rep, torch.float32)
        o = out or dict(accept_len=self._empty((R,), torch.int32),
                        next_token=self._empty((R,), torch.int32))
        dsd_verify_gated(self.handle, R, P, U, E, W, gated_rep, prev_tok, tokens, lse_q,
                         logit_at_tok, keep_len, req_id, temperature, seed, o["accept_len"],
                         o["next_token"], stream, self.device)
        return o

    def propose_rnn(self, U, E, W, h, W_rnn, conf, prev_tok, req_id=None, temperature=0.0,
                    seed=0, out=None, stream=None):
        """dsd_propose with the RNN head; h [R, gamma, H], W_rnn
        [3, rank, 2 rank + H].  Also returns rnn_rep [R, gamma, rank] f32."""
        R, G, H = h.shape
        for n, t in (("U", U), ("E", E), ("W", W), ("h", h), ("W_rnn", W_rnn)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("conf", conf, torch.float32)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("req_id", req_id, torch.int32)
        o = out or dict(tokens=self._empty((R, G), torch.int32),
                        lse_q=self._empty((R, G), torch.float32),
                        logit_at_tok=self._empty((R, G), torch.float32),
                        survival=self._empty((R, G), torch.float32),
                        rnn_rep=self._empty((R, G, self.rank), torch.float32))
        dsd_propose_rnn(self.handle, R, U, E, W, h, H, W_rnn, conf, prev_tok, req_id, temperature,
                        seed, o["tokens"], o["lse_q"], o["logit_at_tok"], o["survival"],
                        o["rnn_rep"], stream, self.device)
        return o

    def verify_rnn(self, P, tokens, keep_len, rnn_rep=None, U=None, E=None, W=None,
                   prev_tok=None, lse_q=None, logit_at_tok=None, req_id=None, temperature=0.0,
                   seed=0, out=None, stream=None):
        R = P.shape[0]
        self._check_in("P", P, self.torch_dtype)
        self._check_in("tokens", tokens, torch.int32)
        self._check_in("keep_len", keep_len, torch.int32)
        self._check_in("rnn_rep", rnn_rep, torch.float32)
        o = out or dict(accept_len=self._empty((R,), torch.int32),
                        next_token=self._empty((R,), torch.int32))
        dsd_verify_rnn(self.handle, R, P, U, E, W, rnn_rep, prev_tok, tokens, lse_q,
                       logit_at_tok, keep_len, req_id, temperature, seed, o["accept_len"],
                       o["next_token"], stream, self.device)
        return o

    def schedule(self, survival, sps, out=None, stream=None):
        R = survival.shape[0]
        self._check_in("survival", survival, torch.float32)
        self._check_in("sps", sps, torch.float32)
        o = out or dict(keep_len=self._empty((R,), torch.int32),
                        theta_B=self._empty((2,), torch.float32))
        dsd_schedule(self.handle, R, survival, sps, sps.numel(), o["keep_len"], o["theta_B"],
                     stream, self.device)
        return o

    def verify(self, P, tokens, keep_len, U=None, E=None, W=None, prev_tok=None, lse_q=None,
               logit_at_tok=None, req_id=None, temperature=0.0, seed=0, out=None, stream=None):
        R = P.shape[0]
        self._check_in("P", P, self.torch_dtype)
        self._check_in("tokens", tokens, torch.int32)
        self._check_in("keep_len", keep_len, torch.int32)
        o = out or dict(accept_len=self._empty((R,), torch.int32),
                        next_token=self._empty((R,), torch.int32))
        dsd_verify(self.handle, R, P, U, E, W, prev_tok, tokens, lse_q, logit_at_tok, keep_len,
                   req_id, temperature, seed, o["accept_len"], o["next_token"], stream,
                   self.device)
        return o

    def cycle_outputs(self, R):
        G = self.gamma
        return dict(tokens=self._empty((R, G), torch.int32),
                    lse_q=self._empty((R, G), torch.float32),
                    logit_at_tok=self._empty((R, G), torch.float32),
                    survival=self._empty((R, G), torch.float32),
                    keep_len=self._empty((R,), torch.int32),
                    theta_B=self._empty((2,), torch.float32),
                    accept_len=self._empty((R,), torch.int32),
                    next_token=self._empty((R,), torch.int32))

    def cycle(self, U, E, W, conf, prev_tok, P, sps, req_id=None, temperature=0.0, seed=0,
              out=None, stream=None):
        R = U.shape[0]
        o = out or self.cycle_outputs(R)
        dsd_cycle(self.handle, R, U, E, W, conf, prev_tok, req_id, P, sps, sps.numel(),
                  temperature, seed, o["tokens"], o["lse_q"], o["logit_at_tok"], o["survival"],
                  o["keep_len"], o["theta_B"], o["accept_len"], o["next_token"], stream,
                  self.device)
        return o

    def cycle_host(self, U_host, E, W, conf_host, prev_tok_host, P_host, sps, req_id_host=None,
                   temperature=0.0, seed=0, out=None, stream=None):
        """One cycle from host tensors (pinned for asynchronous copies)."""
        R = U_host.shape[0]
        G = self.gamma
        o = out or dict(tokens=torch.empty((R, G), dtype=torch.int32, pin_memory=True),
                        keep_len=torch.empty((R,), dtype=torch.int32, pin_memory=True),
                        accept_len=torch.empty((R,), dtype=torch.int32, pin_memory=True),
                        next_token=torch.empty((R,), dtype=torch.int32, pin_memory=True))
        dsd_cycle_host(self.handle, R, U_host, E, W, conf_host, prev_tok_host, req_id_host,
                       P_host, sps, sps.numel(), temperature, seed, o["tokens"], o["keep_len"],
                       o["accept_len"], o["next_token"], stream, self.device)
        return o

    def overlap(self, P_logits, Q_logits, valid_len, out=None, stream=None):
        N = P_logits.shape[0]
        self._check_in("P_logits", P_logits, self.torch_dtype)
        self._check_in("Q_logits", Q_logits, self.torch_dtype)
        self._check_in("valid_len", valid_len, torch.int32)
        G = self.gamma
        o = out or dict(a=self._empty((N, G), torch.float32), l1=self._empty((N, G), torch.float32),
                        tau=self._empty((N,), torch.float32),
                        accept_rate=self._empty((G,), torch.float32),
                        mean_tau=self._empty((1,), torch.float32))
        dsd_overlap(self.handle, N, P_logits, Q_logits, valid_len, o["a"], o["l1"], o["tau"],
                    o["accept_rate"], o["mean_tau"], stream, self.device)
        return o

    def confidence_head(self, h, E, w_c, b_c, prev_tok, tokens, out=None, stream=None):
        """conf = sigmoid(w_c . [h; E[t_prev]] + b_c) and its prefix survival,
        both [R, gamma] f32.  h is [R, gamma, H]."""
        R, G, H = h.shape
        for n, t in (("h", h), ("E", E), ("w_c", w_c)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("tokens", tokens, torch.int32)
        o = out or dict(conf=self._empty((R, G), torch.float32),
                        survival=self._empty((R, G), torch.float32))
        dsd_confidence_head(self.handle, R, H, h, E, w_c, float(b_c), prev_tok, tokens, o["conf"],
                            o["survival"], stream, self.device)
        return o

    def threshold_keep(self, conf, threshold, out=None, stream=None):
        """keep_len [R] i32: leading positions with conf >= threshold."""
        self._check_in("conf", conf, torch.float32)
        keep = out if out is not None else self._empty((conf.shape[0],), torch.int32)
        dsd_threshold_keep(self.handle, conf.shape[0], conf, float(threshold), keep, stream,
                           self.device)
        return keep

    def calibration(self, conf, accept_len, n_bins=10, out=None, stream=None):
        """Reliability bins, per-position survival and (ece, abs_error,
        cumprod_bias, tested positions) of predicted survival against
        realised acceptance."""
        self._check_in("conf", conf, torch.float32)
        self._check_in("accept_len", accept_len, torch.int32)
        o = out or dict(bins=self._empty((3, n_bins), torch.float32),
                        pos=self._empty((2, self.gamma), torch.float32),
                        metrics=self._empty((4,), torch.float32))
        dsd_calibration(self.handle, conf.shape[0], conf, accept_len, n_bins, o["bins"], o["pos"],
                        o["metrics"], stream, self.device)
        return o

    def auroc(self, conf, accept_len, scratch=None, stream=None):
        """AUROC of predicted survival against realised survival (one device
        double).  `scratch` (uint8 device tensor) may be passed to reuse it;
        otherwise it is allocated here, by torch, outside the library."""
        self._check_in("conf", conf, torch.float32)
        self._check_in("accept_len", accept_len, torch.int32)
        M = conf.shape[0]
        need = dsd_auroc_scratch_bytes(M, self.gamma)
        if scratch is None or scratch.numel() < need:
            scratch = torch.empty(need, dtype=torch.uint8, device=self._dev)
        out = self._empty((1,), torch.float64)
        dsd_auroc(self.handle, M, conf, accept_len, scratch, out, stream, self.device)
        return out

    def loss_forward(self, U, E, W, prev_tok, P, target, conf_logit, ce_alpha=0.1, l1_alpha=0.9,
                     conf_alpha=1.0, decay=4.0, rows=True, out=None, stream=None):
        """Teacher-forced DSpark loss forward.  Returns dict(losses=[4] f32:
        ce_loss, l1_loss, conf_loss, total) and, with rows=True, row=[4, B*gamma]
        f32: l1, accept, ce, bce per row n = b * gamma + j."""
        B = U.shape[0]
        for n, t in (("U", U), ("E", E), ("W", W), ("P", P)):
            self._check_in(n, t, self.torch_dtype)
        self._check_in("prev_tok", prev_tok, torch.int32)
        self._check_in("target", target, torch.int32)
        self._check_in("conf_logit", conf_logit, torch.float32)
        o = out or dict(losses=self._empty((4,), torch.float32),
                        row=self._empty((4, B * self.gamma), torch.float32) if rows else None)
        dsd_loss_forward(self.handle, B, U, E, W, prev_tok, P, target, conf_logit, ce_alpha,
                         l1_alpha, conf_alpha, decay, o.get("row"), o["losses"], stream,
                         self.device)
        return o
