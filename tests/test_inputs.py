"""The seeded generators: deterministic, right shapes, the stated
distributions (CPU only)."""

import numpy as np
import torch

from mla_decode_query_gb300 import inputs


def _f(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()


def test_deterministic_and_shapes():
    a = inputs.make_layer(inputs.layer_seed(2, 5), 8, "mxfp8")
    b = inputs.make_layer(inputs.layer_seed(2, 5), 8, "mxfp8")
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    assert a["q_nope"].shape == (32, 8, 128) and a["q_nope"].dtype == np.uint16
    assert a["q_pe"].shape == (32, 8, 64)
    assert a["weight"].shape == (8, 128, 512) and a["weight"].dtype == np.uint8
    assert a["weight_scale"].shape == (8, 128, 16)
    c = inputs.make_layer(inputs.layer_seed(2, 6), 8, "mxfp8")
    assert not np.array_equal(a["weight"], c["weight"])


def test_weights_do_not_depend_on_token_count():
    a = inputs.make_layer(3, 11, "bf16", m_max=32)
    b = inputs.make_layer(3, 11, "bf16", m_max=5)
    np.testing.assert_array_equal(a["weight"], b["weight"])


def test_distributions():
    d = inputs.make_layer(0, 16, "bf16")
    w = _f(d["weight"])
    assert abs(w.std() - 1 / np.sqrt(128)) < 2e-3 and abs(w.mean()) < 1e-3
    q = _f(d["q_nope"])
    assert abs(q.std() - 1) < 0.02
    m = inputs.make_layer(1, 16, "mxfp8")
    s = m["weight_scale"].astype(int)
    assert s.min() == 123 and s.max() == 129
    assert len(np.unique(s)) == 7
    qs = inputs.make_q_scale(3)
    assert qs.dtype == np.float32 and 0.01 <= qs <= 0.1


def test_small_integer_layer_values():
    d = inputs.small_integer_layer(4, 8, 3, "bf16")
    q = _f(d["q_nope"])
    assert set(np.unique(q)) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    w = _f(d["weight"])
    assert set(np.unique(w)) <= {-1.0, 0.0, 1.0}


def test_v_layer_shapes_and_determinism():
    from mla_decode_query_gb300 import inputs as inp
    for fmt in ("bf16", "mxfp8"):
        a = inp.make_v_layer(5, 11, fmt, m_max=7)
        b = inp.make_v_layer(5, 11, fmt, m_max=7)
        assert a["x"].shape == (7, 11, 512) and a["x"].dtype == np.uint16
        assert a["weight"].shape == (11, 512, 128)
        assert a["weight"].dtype == (np.uint16 if fmt == "bf16" else np.uint8)
        for k in ("x", "weight"):
            np.testing.assert_array_equal(a[k], b[k])
        if fmt == "mxfp8":
            s = a["weight_scale"]
            assert s.shape == (11, 512, 4) and s.min() >= 123 and s.max() <= 129
        else:
            assert a["weight_scale"] is None
    w = inp.make_v_layer(6, 16, "bf16")["weight"]
    wf = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert abs(wf.std() * np.sqrt(512) - 1) < 0.02
