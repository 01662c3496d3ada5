"""Thin ctypes binding of libk3moe (include/k3moe.h): argument marshalling only.

PyTorch supplies device memory and streams; every step of the layer runs in
the library's CUDA kernels.  There is no fallback: if the library is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("K3MOE_LIB", os.path.join(_PKG, "libk3moe.so"))

OK = 0
ERR = {0: "OK", -1: "ARG", -2: "SHAPE", -3: "ALIGN", -4: "BAD_SCALE", -5: "ALIAS", -6: "WORKSPACE",
       -7: "CUDA", -8: "TIMEOUT", -9: "UNSUPPORTED", -10: "RANGE", -11: "STATE"}
ERR_CODE = {v: k for k, v in ERR.items()}
PATH_AUTO, PATH_GENERIC, PATH_TENSOR = 0, 1, 2
ROUTER_F32, ROUTER_BF16 = 0, 1
ACT_SILU, ACT_SITU = 0, 1

EXPORTS = ["k3moe_create", "k3moe_persistent_bytes", "k3moe_load_weights", "k3moe_workspace_bytes",
           "k3moe_forward", "k3moe_forward_host", "k3moe_status", "k3moe_destroy", "k3moe_strerror",
           "k3moe_path_for", "k3moe_debug_dequant", "k3moe_debug_wait_timeout",
           "k3moe_profile_enable", "k3moe_profile_read", "k3moe_stage_name", "k3moe_qb_workspace_bytes",
           "k3moe_qb_bias", "k3moe_ep_plan_compute", "k3moe_ep_dispatch_workspace_bytes", "k3moe_ep_dispatch",
           "k3moe_route_static", "k3moe_mma_peak"]
STAGES = ["router", "down_proj", "topk", "permute", "gate_up", "expert_down", "combine_norm",
          "up_proj", "shared", "finish", "prep", "shared_down"]


class K3Error(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"k3moe error {code} ({ERR.get(code, '?')}) {what}")


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("latent", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
                ("inter", C.c_int), ("shared_inter", C.c_int), ("rms_eps", C.c_float),
                ("routed_scaling", C.c_float), ("act", C.c_int), ("router_dtype", C.c_int),
                ("has_select_bias", C.c_int), ("path", C.c_int), ("situ_beta", C.c_float),
                ("situ_linear_beta", C.c_float), ("a8", C.c_int)]


_PP = C.POINTER(C.c_void_p)


class Weights(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("select_bias", C.c_void_p), ("w_down", C.c_void_p),
                ("w_up", C.c_void_p), ("norm_gamma", C.c_void_p),
                ("w1_packed", _PP), ("w1_scale", _PP), ("w3_packed", _PP), ("w3_scale", _PP),
                ("w2_packed", _PP), ("w2_scale", _PP),
                ("ws1_packed", C.c_void_p), ("ws1_scale", C.c_void_p), ("ws3_packed", C.c_void_p),
                ("ws3_scale", C.c_void_p), ("ws2_packed", C.c_void_p), ("ws2_scale", C.c_void_p)]


_lib = None


class EpPlan(C.Structure):
    """k3moe_ep_plan: device pointers of a balanced expert-parallel plan."""
    _fields_ = [("seg", C.c_void_p), ("rank_seg", C.c_void_p), ("exp_off", C.c_void_p),
                ("exp_seg", C.c_void_p), ("info", C.c_void_p)]


def lib():
    """Load libk3moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                              "(python latent_moe_layer_gb300/build.py)")
        L = C.CDLL(LIB_PATH)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        L.k3moe_create.argtypes = [C.POINTER(Config), C.POINTER(vp)]
        L.k3moe_persistent_bytes.argtypes = [vp]
        L.k3moe_persistent_bytes.restype = sz
        L.k3moe_load_weights.argtypes = [vp, C.POINTER(Weights), vp, sz, vp]
        L.k3moe_workspace_bytes.argtypes = [vp, i]
        L.k3moe_workspace_bytes.restype = sz
        L.k3moe_forward.argtypes = [vp, vp, i, vp, vp, vp, vp, sz, vp]
        L.k3moe_forward_host.argtypes = [vp, vp, i, vp, vp, vp, vp, sz, vp]
        L.k3moe_status.argtypes = [vp, vp]
        L.k3moe_destroy.argtypes = [vp]
        L.k3moe_destroy.restype = None
        L.k3moe_strerror.argtypes = [i]
        L.k3moe_strerror.restype = C.c_char_p
        L.k3moe_path_for.argtypes = [vp, i]
        L.k3moe_debug_dequant.argtypes = [vp, vp, i, i, vp, vp]
        L.k3moe_debug_wait_timeout.argtypes = [vp, i, vp]
        L.k3moe_profile_enable.argtypes = [vp, i]
        L.k3moe_profile_read.argtypes = [vp, vp, vp, vp]
        L.k3moe_stage_name.argtypes = [i]
        L.k3moe_stage_name.restype = C.c_char_p
        L.k3moe_qb_workspace_bytes.argtypes = [vp, i, i]
        L.k3moe_qb_workspace_bytes.restype = sz
        L.k3moe_qb_bias.argtypes = [vp, vp, i, vp, vp, i, vp, sz, vp]
        L.k3moe_ep_plan_compute.argtypes = [vp, vp, i, i, C.POINTER(EpPlan), vp]
        L.k3moe_ep_dispatch_workspace_bytes.argtypes = [vp, i]
        L.k3moe_ep_dispatch_workspace_bytes.restype = sz
        L.k3moe_ep_dispatch.argtypes = [vp, vp, i, i, vp, i, C.POINTER(EpPlan), vp, vp, vp, sz, vp]
        L.k3moe_route_static.argtypes = [vp, vp, i, vp, vp, vp]
        L.k3moe_mma_peak.argtypes = [i, i, i, vp, C.POINTER(C.c_float), vp]
        for name in EXPORTS:
            getattr(L, name)
        _lib = L
    return _lib


def check(rc, what=""):
    if rc != OK:
        raise K3Error(rc, what)


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def make_config(cfg, path=PATH_AUTO) -> Config:
    """k3moe_config from a synth.LayerConfig (or anything with the same fields)."""
    act = {"silu": ACT_SILU, "situ": ACT_SITU}[getattr(cfg, "act", "silu")]
    return Config(cfg.H, cfg.L, cfg.E, cfg.K, cfg.I, cfg.S, cfg.rms_eps, cfg.routed_scaling, act,
                  ROUTER_BF16 if cfg.router_dtype == "bf16" else ROUTER_F32,
                  1 if cfg.select_bias else 0, path, getattr(cfg, "situ_beta", 4.0),
                  getattr(cfg, "situ_linear_beta", 25.0), 1 if getattr(cfg, "a8", False) else 0)


class Layer:
    """One k3moe handle plus its persistent buffer (torch-allocated)."""

    def __init__(self, cfg, path=PATH_AUTO):
        import torch
        self.cfg = cfg
        self.ccfg = make_config(cfg, path)
        h = C.c_void_p()
        check(lib().k3moe_create(C.byref(self.ccfg), C.byref(h)), "create")
        self.h = h
        nb = lib().k3moe_persistent_bytes(self.h)
        self.persist = torch.empty(nb + 256, dtype=torch.uint8, device="cuda")
        self._keep = None
        self._ws = None

    def __del__(self):
        try:
            if getattr(self, "h", None):
                lib().k3moe_destroy(self.h)
                self.h = None
        except Exception:
            pass

    def load(self, dw, stream=None):
        """Record device weights (a DeviceWeights)."""
        E = self.cfg.E
        arr = lambda ptrs: (C.c_void_p * E)(*ptrs)
        tabs = [arr(dw.expert_ptrs(m, part)) for m in range(3) for part in range(2)]
        sh = [None] * 6
        if self.cfg.S:
            sh = [_ptr(dw.shared[m][part]) for m in range(3) for part in range(2)]
        pp = lambda t: C.cast(t, _PP)
        w = Weights(_ptr(dw.w_router), _ptr(dw.bias), _ptr(dw.w_down), _ptr(dw.w_up), _ptr(dw.gamma),
                    pp(tabs[0]), pp(tabs[1]), pp(tabs[2]), pp(tabs[3]), pp(tabs[4]), pp(tabs[5]), *sh)
        base = self.persist.data_ptr()
        aligned = (base + 255) // 256 * 256
        rc = lib().k3moe_load_weights(self.h, C.byref(w), aligned,
                                      self.persist.numel() - (aligned - base), _stream_ptr(stream))
        check(rc, "load_weights")
        self._keep = (dw, tabs, w)

    def path_for(self, T):
        return lib().k3moe_path_for(self.h, T)

    def workspace_bytes(self, T):
        return lib().k3moe_workspace_bytes(self.h, T)

    def workspace(self, T):
        import torch
        nb = self.workspace_bytes(T)
        if self._ws is None or self._ws.numel() < nb:
            self._ws = None
            self._ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        return self._ws

    def forward(self, x, out=None, idx_out=None, w_out=None, workspace=None, stream=None):
        """x: [T, H] bf16 CUDA tensor -> out [T, H] bf16 (async on the stream)."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        ws = workspace if workspace is not None else self.workspace(T)
        rc = lib().k3moe_forward(self.h, _ptr(x), T, _ptr(out), _ptr(idx_out), _ptr(w_out), _ptr(ws),
                                 ws.numel(), _stream_ptr(stream))
        check(rc, "forward")
        return out

    def forward_host(self, x_host, out_host, idx_host=None, w_host=None, workspace=None, stream=None):
        """Host-buffer forward (pinned CPU tensors); synchronises before returning."""
        T = x_host.shape[0]
        ws = workspace if workspace is not None else self.workspace(T)
        rc = lib().k3moe_forward_host(self.h, _ptr(x_host), T, _ptr(out_host), _ptr(idx_host),
                                      _ptr(w_host), _ptr(ws), ws.numel(), _stream_ptr(stream))
        check(rc, "forward_host")
        return out_host

    def status(self, stream=None):
        return lib().k3moe_status(self.h, _stream_ptr(stream))

    def profile(self, enable=True):
        check(lib().k3moe_profile_enable(self.h, 1 if enable else 0), "profile_enable")

    def profile_read(self, stream=None):
        """-> (forwards covered, {stage: ms summed}, {stage: kernel launches})"""
        n = len(STAGES)
        ms = (C.c_float * n)()
        la = (C.c_int * n)()
        rc = lib().k3moe_profile_read(self.h, ms, la, _stream_ptr(stream))
        if rc < 0:
            check(rc, "profile_read")
        return rc, {STAGES[i]: ms[i] for i in range(n)}, {STAGES[i]: la[i] for i in range(n)}

    def qb_bias(self, logits, bias_in=None, nbins=1000, stream=None):
        """Quantile-Balancing bias update from router logits (fp32 CUDA [T, E]) -> fp32 [E]."""
        import torch
        T = logits.shape[0]
        n = lib().k3moe_qb_workspace_bytes(self.h, T, nbins)
        if n == 0:
            raise K3Error(ERR_CODE["ARG"], "qb_workspace_bytes")
        ws = torch.empty(n, dtype=torch.uint8, device=logits.device)
        out = torch.empty(logits.shape[1], dtype=torch.float32, device=logits.device)
        check(lib().k3moe_qb_bias(self.h, logits.data_ptr(), T, _ptr(bias_in), out.data_ptr(), nbins,
                                  ws.data_ptr(), n, _stream_ptr(stream)), "qb_bias")
        return out

    def ep_plan(self, counts, tokens_per_rank, out=None, stream=None):
        """Balanced expert-parallel plan from all ranks' per-expert counts (int32
        CUDA [R, E]) -> dict of int32 CUDA tensors seg [2E, 5] (expert, rank,
        src, count, dst), rank_seg [R, 2], exp_off [E + 1], exp_seg [2E], info [2]
        (written into `out`, such a dict, when given)."""
        import torch
        R, E = counts.shape
        dev = counts.device
        plan = out if out is not None else dict(
            seg=torch.empty((2 * E, 5), dtype=torch.int32, device=dev),
            rank_seg=torch.empty((R, 2), dtype=torch.int32, device=dev),
            exp_off=torch.empty(E + 1, dtype=torch.int32, device=dev),
            exp_seg=torch.empty(2 * E, dtype=torch.int32, device=dev),
            info=torch.empty(2, dtype=torch.int32, device=dev))
        check(lib().k3moe_ep_plan_compute(self.h, counts.data_ptr(), R, tokens_per_rank,
                                          C.byref(_ep_struct(plan)), _stream_ptr(stream)), "ep_plan")
        return plan

    def ep_dispatch(self, idx, src_rank, counts, plan, out=None, workspace=None, stream=None):
        """Destinations (rank, row) of source rank src_rank's routed pairs idx
        (int32 CUDA [S, K]) under `plan` -> two int32 CUDA tensors [S, K]
        (written into `out`, a pair of such tensors, when given; `workspace` a
        uint8 CUDA tensor of ep_dispatch_workspace_bytes(S) bytes)."""
        import torch
        S = idx.shape[0]
        n = lib().k3moe_ep_dispatch_workspace_bytes(self.h, S)
        if n == 0:
            raise K3Error(ERR_CODE["ARG"], "ep_dispatch_workspace_bytes")
        if workspace is not None and workspace.numel() >= n:
            ws, n = workspace, workspace.numel()
        else:
            ws = torch.empty(n, dtype=torch.uint8, device=idx.device)
        rank, row = out if out is not None else (torch.empty_like(idx), torch.empty_like(idx))
        check(lib().k3moe_ep_dispatch(self.h, idx.data_ptr(), S, src_rank, counts.data_ptr(), counts.shape[0],
                                      C.byref(_ep_struct(plan)), rank.data_ptr(), row.data_ptr(), ws.data_ptr(), n,
                                      _stream_ptr(stream)), "ep_dispatch")
        return rank, row

    def ep_dispatch_workspace_bytes(self, tokens_per_rank):
        return lib().k3moe_ep_dispatch_workspace_bytes(self.h, tokens_per_rank)

    def debug_wait_timeout(self, spin_limit, stream=None):
        check(lib().k3moe_debug_wait_timeout(self.h, spin_limit, _stream_ptr(stream)), "wait")


MMA_KINDS = {"f16": 0, "mxf8f6f4_e4m3": 1, "mxf8f6f4_e2m1_e4m3": 2}


def mma_peak(kind, n=256, iters=4096, stream=None):
    """TFLOP/s of back-to-back tcgen05.mma of `kind` (a MMA_KINDS key), M 128, N n, on all SMs."""
    import torch
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    ms = C.c_float()
    check(lib().k3moe_mma_peak(MMA_KINDS[kind], n, iters, status.data_ptr(), C.byref(ms), _stream_ptr(stream)),
          "mma_peak")
    if int(status[0]) != 0:
        raise K3Error(int(status[0]), "mma_peak")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * iters * 2.0 * 128 * n * 128 / (ms.value * 1e-3) / 1e12


def _ep_struct(plan):
    return EpPlan(plan["seg"].data_ptr(), plan["rank_seg"].data_ptr(), plan["exp_off"].data_ptr(),
                  plan["exp_seg"].data_ptr(), plan["info"].data_ptr())


def debug_dequant(packed, scale, stream=None):
    """Decode an MXFP4 matrix on the device (packed/scale uint8 CUDA tensors) -> fp32 tensor."""
    import torch
    rows, cols = packed.shape[0], packed.shape[1] * 2
    out = torch.empty((rows, cols), dtype=torch.float32, device=packed.device)
    check(lib().k3moe_debug_dequant(_ptr(packed), _ptr(scale), rows, cols, _ptr(out),
                                    _stream_ptr(stream)), "dequant")
    return out


class DeviceWeights:
    """Layer weights in device memory (torch tensors), drawn by the seeded generator.

    Experts are stored stacked per matrix ([E, rows, cols/2] packed, [E, rows,
    cols/32] scale) and handed to the library as per-expert pointers, the
    layout the checkpoint's shard header uses for each expert tensor.
    """

    def __init__(self, cfg, dense=None, experts=None, threads=16, batch=32):
        import torch
        from . import synth
        self.cfg = cfg
        d = dense if dense is not None else synth.gen_dense(cfg)
        self.dense = d
        dev = "cuda"
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        if cfg.router_dtype == "bf16":
            self.w_router = t(d.w_router.view(np.int16))
        else:
            self.w_router = t(d.w_router)
        self.bias = t(d.select_bias) if d.select_bias is not None else None
        self.w_down = t(d.w_down.view(np.int16))
        self.w_up = t(d.w_up.view(np.int16))
        self.gamma = t(d.gamma.view(np.int16))
        self.shared = None
        if cfg.S and d.shared is not None:
            self.shared = [(t(p), t(s)) for p, s in d.shared]
        dims = synth.expert_dims(cfg)
        self.packed, self.scale = [], []
        for (r, c) in dims:
            self.packed.append(torch.empty((cfg.E, r, c // 2), dtype=torch.uint8, device=dev))
            self.scale.append(torch.empty((cfg.E, r, c // 32), dtype=torch.uint8, device=dev))
        if experts is not None:   # explicit host experts {e: [(p, s)] * 3}
            for e in range(cfg.E):
                for m, (p, s) in enumerate(experts[e]):
                    self.packed[m][e].copy_(torch.from_numpy(p))
                    self.scale[m][e].copy_(torch.from_numpy(s))
        else:
            self._upload_generated(threads, batch)
        torch.cuda.synchronize()

    def _upload_generated(self, threads, batch):
        import torch
        from . import synth
        cfg = self.cfg
        dims = synth.expert_dims(cfg)
        nb = min(batch, cfg.E)
        stp = [torch.empty((nb, r, c // 2), dtype=torch.uint8).pin_memory() for r, c in dims]
        sts = [torch.empty((nb, r, c // 32), dtype=torch.uint8).pin_memory() for r, c in dims]
        pn = [s.numpy() for s in stp]
        sn = [s.numpy() for s in sts]
        for e0 in range(0, cfg.E, nb):
            n = min(nb, cfg.E - e0)
            torch.cuda.synchronize()          # staging reuse
            synth.gen_experts_into(cfg, [_Offset(a, e0) for a in pn], [_Offset(a, e0) for a in sn],
                                   experts=range(e0, e0 + n), threads=threads)
            for m in range(3):
                self.packed[m][e0:e0 + n].copy_(stp[m][:n], non_blocking=True)
                self.scale[m][e0:e0 + n].copy_(sts[m][:n], non_blocking=True)

    def expert_ptrs(self, m, part):
        t = self.packed[m] if part == 0 else self.scale[m]
        step = t.stride(0) * t.element_size()
        base = t.data_ptr()
        return [base + e * step for e in range(self.cfg.E)]


class _Offset:
    """Index shim: a[e] -> base[e - e0] (lets the generator fill a batch buffer)."""

    def __init__(self, base, e0):
        self.base, self.e0 = base, e0

    def __setitem__(self, e, v):
        self.base[e - self.e0] = v
