"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot allocate
device memory (a host framework owning all device memory, a path that must not
make the device synchronise, a plugin host that forbids allocation), against
moe_dispatch and against the oracle's dispatch.  Collected last on purpose: it shares
one library-wide scratch array, so it is run after (and also works without) every
other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import _lib, api, configs
from support import bf16_dev, host_workload, to_dev, unpack_sf_atoms

pytestmark = pytest.mark.gpu


def _outputs(cfg, B, dev):
    sz = api.dispatch_sizes(cfg, B)
    rows, mt = sz["rows"], sz["max_tiles"]
    srows = (B + 127) // 128 * 128
    e = lambda *s, dt=torch.uint8: torch.full(s, 0x5A, dtype=dt, device=dev) if dt == torch.uint8 \
        else torch.full(s, -7, dtype=dt, device=dev)  # noqa: E731
    return dict(A=e(rows, cfg.H), A_sf=e(api.scale_bytes(rows, cfg.H)),
                counts=e(cfg.N_phys, dt=torch.int32), row_of=e(B, cfg.K, dt=torch.int32),
                src_of=e(rows, dt=torch.int32), tiles=e(8 + 16 * mt, dt=torch.int32),
                As=e(srows, cfg.H), As_sf=e(api.scale_bytes(srows, cfg.H)),
                shared_tiles=e(8 + 16 * (srows // 128), dt=torch.int32),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _call(fn_name, cfg, x, idx, l2p, rep, o, ws=None):
    L = _lib.load()
    dc = _lib.DispatchCfg(x.shape[0], cfg.H, cfg.K, cfg.N, cfg.N_phys, cfg.layout, cfg.cap, 0)
    p = _lib.ptr
    args = [ctypes.byref(dc), p(x), p(idx), p(l2p), p(rep), p(o["A"]), p(o["A_sf"]),
            p(o["counts"]), p(o["row_of"]), p(o["src_of"]), p(o["tiles"]), p(o["As"]),
            p(o["As_sf"]), p(o["shared_tiles"])]
    if ws is not None:
        args += [p(ws), ws.numel()]
    args += [p(o["status"]), _lib.stream_ptr()]
    _lib.check(getattr(L, fn_name)(*args), fn_name)


def _valid_equal(cfg, a, b):
    """Equal on everything the dispatch defines (padding rows are never written)."""
    for k in ("counts", "row_of", "src_of", "tiles", "status"):
        assert torch.equal(a[k], b[k]), k
    ro = a["row_of"].reshape(-1)
    rows = ro[ro >= 0].long()
    assert torch.equal(a["A"][rows], b["A"][rows])
    kb = cfg.H // 128
    sfa = unpack_sf_atoms(a["A_sf"].cpu().numpy(), a["A"].shape[0], kb)
    sfb = unpack_sf_atoms(b["A_sf"].cpu().numpy(), b["A"].shape[0], kb)
    r = rows.cpu().numpy()
    assert np.array_equal(sfa[r], sfb[r])
    B = a["row_of"].shape[0]
    assert torch.equal(a["As"][:B], b["As"][:B])


@pytest.mark.parametrize("names", [("small_eplb", "decode"), ("sbo", "small_contig")])
def test_noalloc_matches_dispatch_on_two_calls_in_a_row(dev, names):
    for name in names:                       # two calls in a row share the scratch array
        cfg, x, W, bias = host_workload(name)
        idx, _ = oracle.route(x, W, bias, cfg)
        l2p = rep = None
        if cfg.N_phys != cfg.N:
            l2p, rep, _ = oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N,
                                                cfg.N_phys)
        xd, idd, l2d, repd = bf16_dev(x), to_dev(idx), to_dev(l2p), to_dev(rep)
        ref = _outputs(cfg, cfg.B, dev)
        ws = torch.empty(api.dispatch_sizes(cfg)["ws"], dtype=torch.uint8, device=dev)
        _call("moe_dispatch", cfg, xd, idd, l2d, repd, ref, ws)
        got = _outputs(cfg, cfg.B, dev)
        _call("moe_dispatch_noalloc", cfg, xd, idd, l2d, repd, got)
        torch.cuda.synchronize()
        _valid_equal(cfg, ref, got)
        _oracle_equal(cfg, x, idx, l2p, rep, got)


def _oracle_equal(cfg, x, idx, l2p, rep, got):
    """The allocation-free call's output against the oracle's dispatch, bit for bit."""
    o = oracle.dispatch(x, idx, cfg, log2phys=l2p, rep=rep)
    assert np.array_equal(got["counts"].cpu().numpy(), o["cnt"])
    ro = got["row_of"].cpu().numpy()
    assert np.array_equal(ro, o["row_of"])
    rows = got["A"].shape[0]
    assert np.array_equal(got["src_of"].cpu().numpy(), o["src_of"][:rows])
    v = ro[ro >= 0]
    assert np.array_equal(got["A"].cpu().numpy()[v], o["A"][v])
    sf = unpack_sf_atoms(got["A_sf"].cpu().numpy(), rows, cfg.H // 128)
    assert np.array_equal(sf[v], o["sf"][v])
    assert got["status"].item() == (1 if o["dropped"] else 0)


def test_noalloc_rejects_sizes_beyond_its_scratch(dev):
    cfg = configs.PREFILL.with_(B=65536, K=16)       # needs more than 4 MiB of scratch
    need = api.dispatch_sizes(cfg)["ws"]
    assert need > (4 << 20)
    dc = _lib.DispatchCfg(cfg.B, cfg.H, cfg.K, cfg.N, cfg.N_phys, cfg.layout, cfg.cap, 0)
    rc = _lib.load().moe_dispatch_noalloc(ctypes.byref(dc), *([None] * 15))
    assert rc == -2                                   # MOE_ERR_UNSUPPORTED, nothing launched
