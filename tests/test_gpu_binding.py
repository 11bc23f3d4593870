"""The Python binding refuses tensors whose dtype, shape or device does not
match the C ABI's layout before anything is launched."""

import pytest
import torch

import paged_kv_cache_202_gb300 as pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def t():
    B, Hq, Hkv, D, bs, NB, MB = 2, 8, 2, 128, 16, 16, 4
    bf = torch.bfloat16
    return dict(q=torch.zeros(B, Hq, D, dtype=bf, device="cuda"),
                k=torch.zeros(NB, Hkv, bs, D, dtype=bf, device="cuda"),
                v=torch.zeros(NB, Hkv, bs, D, dtype=bf, device="cuda"),
                bt=torch.zeros(B, MB, dtype=torch.int32, device="cuda"),
                sl=torch.ones(B, dtype=torch.int32, device="cuda"),
                qs=torch.arange(B + 1, dtype=torch.int32, device="cuda"),
                out=torch.zeros(B, Hq, D, dtype=bf, device="cuda"),
                kn=torch.zeros(B, Hkv, D, dtype=bf, device="cuda"))


def _decode(t, plan, **kw):
    a = dict(t)
    a.update(kw)
    return pa.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["sl"], 0.1, a["out"], 64, plan)


@pytest.mark.parametrize("kw,exc", [
    (dict(bt="int64"), TypeError),
    (dict(sl="int64"), TypeError),
    (dict(sl="short"), ValueError),
    (dict(bt="short"), ValueError),
    (dict(q="f32"), TypeError),
    (dict(out="short"), ValueError),
    (dict(v="short"), ValueError),
    (dict(sl="host"), ValueError),
])
def test_decode_rejects_mismatched_tensors(t, kw, exc):
    key, how = next(iter(kw.items()))
    x = t[key]
    bad = {"int64": lambda: x.long(), "short": lambda: x[:-1].contiguous(),
           "f32": lambda: x.float(), "host": lambda: x.cpu()}[how]()
    plan = pa.Plan()
    with pytest.raises(exc):
        _decode(t, plan, **{key: bad})
    assert plan.handle.value is None, "a refused call must not create a plan"


def test_decode_multi_and_append_check_their_index_tensors(t):
    plan = pa.Plan()
    with pytest.raises(ValueError):   # q_start needs B + 1 entries
        pa.pa_decode_multi(t["q"], t["qs"][:-1].contiguous(), t["k"], t["v"], t["bt"], t["sl"],
                           0.1, t["out"], 1, 64, plan)
    with pytest.raises(TypeError):
        pa.pa_append_kv(t["kn"], t["kn"], t["k"], t["v"], t["bt"], t["sl"].long())
    with pytest.raises(ValueError):   # one new token per sequence and kv head
        pa.pa_append_kv(t["kn"][:1].contiguous(), t["kn"], t["k"], t["v"], t["bt"], t["sl"])
    assert plan.handle.value is None
