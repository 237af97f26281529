"""tree_gemm and tree_rmsnorm (include/tree_layer.h) against the float64 oracle."""
import numpy as np
import pytest

import prefix_tree_packed_gb300 as lib
from oracle import layer as ol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _ulp16(x):
    return np.spacing(np.abs(np.asarray(x, np.float16))).astype(np.float64)


def _close16(got, ref, extra=0.0):
    """At most one f16 ulp of the reference apart (plus `extra` absolute)."""
    g = np.asarray(got, np.float16).astype(np.float64)
    r = np.asarray(ref, np.float16).astype(np.float64)
    bad = np.abs(g - r) > _ulp16(r) + extra
    assert not bad.any(), f"{int(bad.sum())} elements off; worst {np.abs(g - r).max():.3g}"


def _inputs(m, n_b, k, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((m, k)).astype(np.float16)
    b = (rng.standard_normal((n_b, k)) / np.sqrt(k)).astype(np.float16)
    r = rng.standard_normal((m, n_b)).astype(np.float16)
    return a, b, r


SHAPES = [(128, 256, 64), (300, 264, 136), (1000, 768, 520), (2048, 3072, 2048), (77, 8, 8), (129, 520, 4096)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("epi", ["store", "residual", "swiglu"])
def test_gemm_matches_oracle(m, n, k, epi):
    dev = torch.device("cuda")
    n_b = 2 * n if epi == "swiglu" else n
    a, b, r = _inputs(m, n_b, k, seed=m + n + k)
    r = r[:, :n].copy()
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    tr = torch.from_numpy(r).to(dev)
    tc = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    code = {"store": lib.GEMM_STORE, "residual": lib.GEMM_RESIDUAL, "swiglu": lib.GEMM_SWIGLU}[epi]
    lib.gemm(ta, tb, tc, m, n, k, code, r=tr if epi == "residual" else None, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = ol.gemm(a, b, epi, r)
    # f32 accumulation against float64: one f16 rounding apart, plus the f32 sum's error
    _close16(tc.cpu().numpy(), ref, extra=1e-4)


def test_gemm_residual_in_place_and_empty():
    dev = torch.device("cuda")
    a, b, r = _inputs(200, 256, 128, seed=9)
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    tc = torch.from_numpy(r).to(dev)
    lib.gemm(ta, tb, tc, 200, 256, 128, lib.GEMM_RESIDUAL, r=tc)   # C = A B^T + C
    torch.cuda.synchronize()
    _close16(tc.cpu().numpy(), ol.gemm(a, b, "residual", r), extra=1e-4)
    lib.gemm(ta, tb, tc, 0, 256, 128)  # m = 0: nothing to do


def test_gemm_argument_checks():
    dev = torch.device("cuda")
    x = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 60, 64)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 64, 64, 7)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 64, 64, lib.GEMM_RESIDUAL)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG


@pytest.mark.parametrize("rows,cols", [(1000, 2048), (3, 8), (257, 4096), (64, 16384)])
def test_rmsnorm_matches_oracle(rows, cols):
    dev = torch.device("cuda")
    rng = np.random.default_rng(rows + cols)
    x = (rng.standard_normal((rows, cols)) * 3).astype(np.float16)
    w = rng.standard_normal(cols).astype(np.float16)
    tx, tw = torch.from_numpy(x).to(dev), torch.from_numpy(w).to(dev)
    ty = torch.empty_like(tx)
    lib.rmsnorm(tx, tw, ty, rows, cols, 1e-5)
    torch.cuda.synchronize()
    ref = ol.rmsnorm(x, w, 1e-5)
    # f32 statistics against float64: the normalised value may round to the other
    # f16 neighbour (one ulp of n), which the weight scales
    n_ulp = _ulp16(ol.f16(ref.astype(np.float64) / np.where(w == 0, 1, w).astype(np.float64)))
    g = ty.cpu().numpy().astype(np.float64)
    r = ref.astype(np.float64)
    assert (np.abs(g - r) <= _ulp16(r) + n_ulp * np.abs(w.astype(np.float64)) + 1e-7).all()
    lib.rmsnorm(tx, tw, tx, rows, cols, 1e-5)   # in place
    torch.cuda.synchronize()
    assert torch.equal(tx, ty)
