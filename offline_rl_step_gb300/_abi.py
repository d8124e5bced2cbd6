"""ctypes declarations of the C ABI in include/ofrl.h (argument marshalling only)."""
import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libofrl.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, ETIMEOUT = 0, -1, -2, -3, -4
HER_FINAL, HER_FUTURE, HER_RANDOM, HER_EPISODE = 0, 1, 2, 3
PREC_FP32, PREC_BF16 = 0, 1
STAT_NONFINITE_GRAD, STAT_BAD_ACTION, STAT_BAD_INDEX, STAT_TIMEOUT, STAT_SANITIZED, STAT_WORDS = 0, 1, 2, 3, 4, 8

vp = C.c_void_p


class Replay(C.Structure):
    _fields_ = [("states", vp), ("next_states", vp), ("actions", vp), ("rewards", vp), ("dones", vp),
                ("episode_ends", vp), ("capacity", C.c_int64), ("num_episodes", C.c_int32),
                ("state_dim", C.c_int32), ("state_stride", C.c_int32), ("goal_dim", C.c_int32)]


class HerCfg(C.Structure):
    _fields_ = [("batch", C.c_int32), ("her_count", C.c_int32), ("strategy", C.c_int32),
                ("goal_threshold", C.c_float), ("seed", C.c_uint64)]


class Batch(C.Structure):
    _fields_ = [("states", vp), ("next_states", vp), ("actions", vp), ("rewards", vp), ("dones", vp),
                ("src_idx", vp), ("donor_idx", vp), ("stride", C.c_int32)]


class VShape(C.Structure):
    _fields_ = [("state_dim", C.c_int32), ("hidden", C.c_int32), ("num_actions", C.c_int32),
                ("prec", C.c_int32)]


class VNet(C.Structure):
    _fields_ = [("params", vp), ("m", vp), ("v", vp), ("t", C.c_int32), ("tau", C.c_float), ("target", vp),
                ("polyak", C.c_float)]


class Opt(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("max_grad_norm", C.c_float), ("beta", C.c_float),
                ("budget", C.c_float * 4), ("alpha", C.c_float * 4), ("weight_clamp_max_abs", C.c_float),
                ("sanitize_sources", C.c_int32)]


# name -> (restype, argtypes)
SIGNATURES = {
    "ofrl_create": (C.c_int32, [C.POINTER(VShape), C.c_int32, C.c_int32, C.POINTER(vp)]),
    "ofrl_destroy": (C.c_int32, [vp]),
    "ofrl_poll_status": (C.c_int32, [vp, vp, C.POINTER(C.c_int32)]),
    "ofrl_status_string": (C.c_char_p, [C.c_int32]),
    "ofrl_workspace_bytes": (C.c_int64, [C.POINTER(VShape), C.c_int32, C.c_int32]),
    "ofrl_her_relabel": (C.c_int32, [vp, C.POINTER(Replay), C.POINTER(HerCfg), C.c_uint64, C.POINTER(Batch), vp]),
    "ofrl_her_relabel_sources": (C.c_int32, [vp, C.POINTER(Replay), C.POINTER(HerCfg), C.c_uint64, vp, vp,
                                             C.POINTER(Batch), vp, vp]),
    "ofrl_episode_ends_append": (C.c_int32, [vp, vp, C.c_int64, C.c_int32, vp, vp, C.c_int32, vp]),
    "ofrl_iql_value_fwd_bwd": (C.c_int32, [vp, vp, vp, C.c_int32, C.c_int32, vp, C.c_float, vp, vp, vp, vp]),
    "ofrl_forward_values": (C.c_int32, [vp, vp, vp, C.c_int32, C.c_int32, vp, vp]),
    "ofrl_iql_target": (C.c_int32, [vp, vp, vp, C.c_int32, vp, vp, C.c_int32, C.c_float, vp, vp, vp]),
    "ofrl_expectile_loss": (C.c_int32, [vp, vp, vp, C.c_int32, C.c_float, vp, vp, vp]),
    "ofrl_adv_weighted_policy": (C.c_int32, [vp, vp, vp, C.c_int32, C.c_int32, C.c_float, vp, vp, vp]),
    "ofrl_budgeted_clip_saxpy": (C.c_int32, [vp, C.POINTER(vp), C.POINTER(C.c_float), C.POINTER(C.c_float),
                                             C.c_int32, C.c_int64, C.c_float, vp, vp, vp]),
    "ofrl_target_ema": (C.c_int32, [vp, vp, C.c_int64, C.c_float, vp]),
    "ofrl_adam_step": (C.c_int32, [vp, vp, vp, vp, vp, C.c_int64, C.c_int32, C.POINTER(Opt), vp, vp]),
    "ofrl_train_step": (C.c_int32, [vp, C.POINTER(Replay), C.POINTER(HerCfg), C.c_uint64, C.POINTER(Batch), vp,
                                    C.POINTER(VNet), C.c_int32, C.POINTER(Opt), C.POINTER(vp), C.c_int32,
                                    vp, vp, vp, vp, vp, vp, vp]),
    "ofrl_train_step_kernels": (C.c_int32, [vp, C.POINTER(Batch), C.c_int32, C.c_int32]),
    "ofrl_select_vnet_path": (C.c_int32, [vp, C.c_int32]),
    "ofrl_vnet_path": (C.c_int32, [vp, C.c_int32]),
    "ofrl_step_graph_create": (C.c_int32, [vp, C.POINTER(Replay), C.POINTER(HerCfg), C.POINTER(Batch), vp, vp,
                                           C.c_int32, C.POINTER(Opt), C.POINTER(vp), C.c_int32, vp, vp, vp, vp, vp,
                                           vp, C.POINTER(vp)]),
    "ofrl_step_graph_launch": (C.c_int32, [vp, C.c_uint64, vp, C.POINTER(vp), vp]),
    "ofrl_step_graph_destroy": (C.c_int32, [vp]),
    "ofrl_step_graph_create_io": (C.c_int32, [vp, C.POINTER(Replay), C.POINTER(HerCfg), C.POINTER(Batch), vp, vp,
                                              C.c_int32, C.POINTER(Opt), C.POINTER(vp), C.c_int32, vp, vp, vp, vp,
                                              vp, vp, vp, vp, vp, C.POINTER(vp)]),
    "ofrl_step_graph_launch_io": (C.c_int32, [vp, C.c_uint64, vp, C.POINTER(vp), vp, vp, vp]),
    "ofrl_noalloc_max_batch": (C.c_int64, [C.POINTER(VShape)]),
    "ofrl_iql_value_fwd_bwd_noalloc": (C.c_int32, [C.POINTER(VShape), vp, vp, C.c_int32, C.c_int32, vp, C.c_float,
                                                   vp, vp, vp, vp]),
    "ofrl_selftest_umma": (C.c_int32, [vp, vp, vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_int32, vp, vp]),
    "ofrl_selftest_barrier": (C.c_int32, [vp, C.c_uint64, C.c_int32]),
    "ofrl_profile_begin": (C.c_int32, [vp, C.c_int32]),
    "ofrl_profile_end": (C.c_int32, [vp, C.POINTER(C.c_float), C.POINTER(C.c_int32)]),
}
PHASES = ("relabel", "vnet", "reduce", "adam")

_LIB = None


class OfrlError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def load(path: str = LIB_PATH):
    """Load libofrl.so (built by offline_rl_step_gb300.build) and declare its symbols."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"the ofrl CUDA library is not built ({path} is missing); run "
            "`python -m offline_rl_step_gb300.build` or __graft_entry__.build() first")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(fn: str, code: int):
    if code != OK:
        msg = load().ofrl_status_string(code).decode()
        raise OfrlError(fn, code, msg)
