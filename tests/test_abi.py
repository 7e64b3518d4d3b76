"""The C ABI library without a GPU: it loads, exports every function the header declares, and its
host-side config checks answer before any CUDA call."""
import ctypes

import pytest

from deepseek_v4_moe_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_exports_every_declared_function(lib):
    names = _lib.declared_functions()
    assert {"moe_ffn_init", "moe_ffn_forward", "moe_ffn_forward_host", "moe_ffn_status", "moe_ffn_debug_copy",
            "moe_ffn_last_error", "moe_ffn_destroy"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def _cfg(**kw):
    base = dict(hidden=256, hc=4, experts=16, top_k=2, inter=128, shared_inter=128, vocab=1024, n_layers=4,
                hash_layer_count=3, max_rows=4, sinkhorn_iters=20, rms_eps=1e-6)
    base.update(kw)
    return _lib.MoeFfnConfig(**base)


def _init(lib, cfg, layers=None):
    arr = (_lib.MoeFfnLayerWeights * max(cfg.n_layers, 1))()
    for l, w in (layers or {}).items():
        for k, v in w.items():
            setattr(arr[l], k, v)
    h = ctypes.c_void_p()
    rc = lib.moe_ffn_init(ctypes.byref(cfg), arr, ctypes.byref(h))
    return rc, lib.moe_ffn_last_error(None).decode()


@pytest.mark.parametrize("bad", [dict(hc=5), dict(hc=0), dict(hidden=200), dict(inter=100), dict(shared_inter=256),
                                 dict(experts=8), dict(experts=1024), dict(top_k=9), dict(top_k=0),
                                 dict(hash_layer_count=5), dict(max_rows=0), dict(vocab=0), dict(sinkhorn_iters=-1),
                                 dict(hidden=16384)])
def test_bad_config(lib, bad):
    rc, msg = _init(lib, _cfg(**bad))
    assert rc == _lib.ERR_BAD_CONFIG, msg


def _fake_layer(**over):
    # Addresses are never dereferenced: the checks that fail here run before any CUDA call.
    w = {n: 0x10000 + 0x100 * i for i, n in enumerate(_lib.WEIGHT_FIELDS)}
    w.update(over)
    return w


def test_missing_routing_source(lib):
    rc, msg = _init(lib, _cfg(), {3: _fake_layer(exp_probs_b=None)})
    assert rc == _lib.ERR_NO_ROUTING_SOURCE, msg
    rc, msg = _init(lib, _cfg(), {0: _fake_layer(tid2eid=None)})
    assert rc == _lib.ERR_NO_ROUTING_SOURCE, msg


def test_partial_weights_and_alignment(lib):
    rc, _ = _init(lib, _cfg(), {3: _fake_layer(gate_exps=None)})
    assert rc == _lib.ERR_NULL_PTR
    rc, _ = _init(lib, _cfg(), {3: _fake_layer(gate=0x10008)})
    assert rc == _lib.ERR_ALIGNMENT


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.moe_ffn_init(None, None, ctypes.byref(h)) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_forward(None, None, None, 1, 0, None, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_status(None) == _lib.ERR_NULL_PTR
    lib.moe_ffn_destroy(None)


def test_experts_may_all_be_left_for_mxfp8(lib):
    # the six bf16 expert matrices NULL together pass the layer checks (the experts come later in
    # MXFP8).  Without a GPU init then stops at the device query; with one it succeeds (at
    # max_rows 4 it reads no weight, so the fake addresses are never touched) and the handle goes.
    exps = dict(gate_exps=None, up_exps=None, down_exps=None, gate_sh=None, up_sh=None, down_sh=None)
    arr = (_lib.MoeFfnLayerWeights * 4)()
    for k, v in _fake_layer(**exps).items():
        setattr(arr[3], k, v)
    h = ctypes.c_void_p()
    rc = lib.moe_ffn_init(ctypes.byref(_cfg()), arr, ctypes.byref(h))
    if rc == _lib.OK:
        lib.moe_ffn_destroy(h)
    assert rc in (_lib.OK, _lib.ERR_CUDA, _lib.ERR_UNSUPPORTED), lib.moe_ffn_last_error(None).decode()
    rc, _ = _init(lib, _cfg(), {3: _fake_layer(gate_exps=None, up_exps=None)})   # some, not all
    assert rc == _lib.ERR_NULL_PTR
    rc, _ = _init(lib, _cfg(), {3: _fake_layer(down_sh=0x10008)})                # present, misaligned
    assert rc == _lib.ERR_ALIGNMENT


def test_new_entry_points_reject_a_null_handle(lib):
    assert lib.moe_ffn_set_attn_hc(None, 0, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_set_mxfp8_experts(None, 0, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_hc_pre(None, 0, 0, None, 1, None, None, None, None, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_hc_post(None, None, None, None, None, 1, None, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_forward_layers(None, None, None, 1, 0, 2, None, None) == _lib.ERR_NULL_PTR
    assert lib.moe_ffn_set_fault_injection(None, 1, 1000) == _lib.ERR_NULL_PTR
