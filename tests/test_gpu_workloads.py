"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark uses (one w4a16_gemm call per (layer, M)).

Repacked words are compared on sampled TILE atoms (every atom is an independent
64 x 16 block), zeros / scales / perm in full. GEMM outputs are compared with
the fp64 oracle on sampled rows (all rows up to M = 64) and sampled columns
(all columns up to N = 16384); rows and columns are independent, so each
sampled output is exact per element. Tolerance: max|y - y_ref| / max|y_ref|
<= 4e-3 over the sample.
"""
import numpy as np
import pytest

import oracle
import synth
from libutil import ensure_built, half_from_dev, half_to_dev, to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-3


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    import int4_weight_only_repack_gb300 as mod
    return mod


def sample_rows(M, rng):
    if M <= 64:
        return np.arange(M)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, 14, replace=False)]))


def sample_cols(N, rng):
    if N <= 16384:
        return np.arange(N)
    return np.unique(np.concatenate([np.arange(1024), np.arange(N - 1024, N),
                                     rng.choice(N, 2048, replace=False)]))


def check_layer(w4, cfg, li):
    import torch
    wl = synth.WORKLOADS[cfg]
    K, N, name = wl.shapes[li]
    L = synth.make_workload_layer(cfg, li)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    qweight, qzeros = to_dev(L.qweight), to_dev(L.qzeros)
    scales = half_to_dev(L.scales, wl.dtype)
    if wl.fmt == "awq":
        layer = w4.repack_awq(qweight, qzeros, scales, K, N, wl.group, dt)
    else:
        layer = w4.repack_gptq(qweight, qzeros, scales, to_dev(L.g_idx), K, N, wl.group, dt)
    del qweight, qzeros, scales
    torch.cuda.synchronize()

    q, z, s = oracle.layer_codes(L.qweight, L.qzeros, L.scales, wl.dtype, wl.fmt)
    rng = np.random.default_rng([7, cfg, li])
    perm = None
    if L.g_idx is not None:
        assert int(layer.status[0].item()) == 0
        perm = oracle.act_order_perm(L.g_idx)
        assert np.array_equal(layer.perm.cpu().numpy(), perm)
    # repack: sampled atoms, bit-exact (atom index: column group, k-atom, tile in group)
    A, NT = K // 64, N // 16
    n_atoms = oracle.tile_words(K, N) // 128
    n_pick = min(n_atoms, 254)
    atoms = np.unique(np.concatenate([[0, n_atoms - 1], rng.choice(n_atoms, n_pick, replace=False)]))
    words = layer.qw.view(-1)
    idx = torch.from_numpy((atoms[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)).to(words.device)
    got = words[idx].cpu().numpy().reshape(len(atoms), 128)
    rows = perm if perm is not None else np.arange(K)
    for i, a in enumerate(atoms):
        cg, rem = divmod(int(a), 8 * A)
        kb, wt = divmod(rem, 8)
        nt = 8 * cg + wt
        if nt >= NT:  # zero padding of the last column group
            assert not got[i].any(), (name, int(a))
            continue
        assert oracle.tile_atom(kb, nt, K) == int(a)
        block = q[rows[64 * kb:64 * kb + 64], 16 * nt:16 * nt + 16]
        assert np.array_equal(got[i], oracle.tile_pack(block)[:128]), (name, int(a))
    zstd = oracle.pack_cols_std(z)
    assert np.array_equal(layer.zeros.cpu().numpy().reshape(zstd.shape), zstd)
    assert np.array_equal(half_from_dev(layer.scales).reshape(L.scales.shape), L.scales)

    # GEMM: dequantise the sampled columns once, reuse for every M
    cols = sample_cols(N, rng)
    gk = oracle.group_of_rows(K, wl.group, L.g_idx)
    W = oracle.dequant(q, z, s, gk, cols=cols).astype(np.float64)
    worst = 0.0
    for M in wl.ms:
        x = synth.make_workload_x(cfg, li, M)
        y = w4.linear(half_to_dev(x, wl.dtype), layer)
        torch.cuda.synchronize()
        r = sample_rows(M, rng)
        y_s = half_from_dev(y[torch.from_numpy(r).to(y.device)][:, torch.from_numpy(cols).to(y.device)])
        y_ref = oracle.gemm(oracle.half_bits_to_f64(x[r], wl.dtype), W)
        err = oracle.rel_err(oracle.half_bits_to_f64(y_s, wl.dtype), y_ref)
        floor = oracle.output_rounding_floor(y_ref, wl.dtype)
        worst = max(worst, err)
        assert err <= TOL, (wl.name, name, M, err, floor)
    return worst


@pytest.mark.parametrize("cfg,li", [(c, l) for c in range(len(synth.WORKLOADS))
                                    for l in range(len(synth.WORKLOADS[c].shapes))])
def test_workload_layer(w4, cfg, li):
    check_layer(w4, cfg, li)
