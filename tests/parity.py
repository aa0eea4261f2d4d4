"""Helpers shared by the GPU parity tests: compare library outputs with the
oracle, with near ties (decisions within 1e-6 relative, recorded by the
oracle) reported instead of silently passed."""

import warnings

import numpy as np

ATTN_TOL = 2e-3     # max abs error of attention outputs (fp32 out, bf16/fp32 inputs)


def report_near_ties(log, what):
    if log:
        warnings.warn(f"{what}: near ties within 1e-6 relative: {log.summary()}")
        return True
    return False


def tree_matches(gpu, ref, what="tree"):
    """Bit-exact comparison of a library Tree with an oracle tree.  If the
    oracle flagged a near tie the structure may legitimately differ: then
    only validity is checked and the tie is reported."""
    m = ref["m"]
    par = gpu.parents.cpu().numpy()
    tok = gpu.tokens.cpu().numpy()
    dep = gpu.depth.cpu().numpy()
    pos = gpu.pos.cpu().numpy()
    mask = gpu.mask_u64()
    if report_near_ties(ref["log"], what):
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, m))
        return False
    np.testing.assert_array_equal(par, ref["parents"], err_msg=f"{what} parents")
    np.testing.assert_array_equal(tok, ref["tokens"], err_msg=f"{what} tokens")
    np.testing.assert_array_equal(dep, ref["depth"], err_msg=f"{what} depth")
    np.testing.assert_array_equal(pos, ref["pos"], err_msg=f"{what} pos")
    np.testing.assert_array_equal(mask, ref["mask"], err_msg=f"{what} mask")
    if gpu.values is not None:
        np.testing.assert_allclose(gpu.values.cpu().numpy(), ref["values"], rtol=0, atol=1e-5,
                                   err_msg=f"{what} values")
    return True


def path_matches(acc, n_acc, bonus, ref, what="verify"):
    n = int(n_acc)
    got_path = list(acc[: n + 1])
    if report_near_ties(ref["log"], what):
        return False
    assert got_path == ref["path"], f"{what}: path {got_path} != {ref['path']}"
    assert int(bonus) == ref["bonus"], f"{what}: bonus {int(bonus)} != {ref['bonus']}"
    return True


def to_device_rows(x, stride=None):
    """Copy fp32 rows [R, V] to the GPU with a row stride that is a multiple of
    4 elements (the library's alignment rule); returns the [R, V] view."""
    import torch
    R, V = x.shape
    stride = stride or (V + 3) // 4 * 4
    full = torch.full((R, stride), -3.0e38, dtype=torch.float32, device="cuda")
    full[:, :V] = x.to("cuda")
    return full[:, :V]


def max_abs(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())
