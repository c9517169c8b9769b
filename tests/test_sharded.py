"""Row-slab sharding of one tensor over ranks.

CPU tests: slab bounds; world-size-2 ``gloo`` ranks (processes) that each
quantize a slab with the oracle as the compute backend and exchange the amax
with a MAX all-reduce, assembled and compared with the oracle run on the
whole tensor (bit-exact); a rank whose slab is invalid (every rank raises,
none waits); a rank that exits before the exchange (the survivor's
collective fails with an error instead of hanging).

GPU test: two host threads play the ranks over slabs of one tensor on the
one GPU (the MAX done on the host between them, no kernel waits on another),
compared with one call on the whole tensor.
"""
import datetime
import os
import pickle
import socket
import threading

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from nvfp4_block_scaled_amax_gb300 import NVFP4Tensor, inputs
from nvfp4_block_scaled_amax_gb300.sharded import (ShardError, assemble, check_slab, quantize_slab,
                                                   slab_alignment, slab_bounds)


# ---------------------------------------------------------------------------
# host logic
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", [0, 1, 15, 16, 127, 128, 1000, 1024, 8192, 8200])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("align", [1, 16, 128])
def test_slab_bounds_partition_the_rows(M, world, align):
    bounds = [slab_bounds(M, world, r, align) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == M
    for (a0, b0), (a1, b1) in zip(bounds, bounds[1:]):
        assert b0 == a1
    for a, b in bounds:
        assert 0 <= a <= b <= M
        assert a % align == 0 or a == b == M
        assert b == M or b % align == 0
    sizes = [-(-(b - a) // align) for a, b in bounds]  # units per rank
    assert max(sizes) - min(sizes) <= 1


def test_slab_alignment_and_checks():
    assert slab_alignment("1d", True, True) == 128
    assert slab_alignment("2d", False, False) == 16
    assert slab_alignment("1d", False, False) == 1
    check_slab(128, 256, "2d", True, True, True)
    check_slab(7, 32, "1d", True, False, False)
    for args in [(8, 32, "1d", True, True, False), (64, 256, "1d", True, True, True),
                 (32, 24, "1d", True, False, False), (32, 32, "row_scaled", True, True, False),
                 (32, 32, "3d", True, True, False)]:
        with pytest.raises(ValueError):
            check_slab(*args)


# ---------------------------------------------------------------------------
# the oracle as the compute backend of a CPU rank (test infrastructure)
# ---------------------------------------------------------------------------

def _bits(x: torch.Tensor) -> np.ndarray:
    if x.dtype == torch.bfloat16:
        return x.contiguous().view(torch.int16).numpy().view(np.uint16)
    return x.contiguous().numpy()


def _to_tensor(d: dict, M: int, N: int, swizzled: bool, row_scaled: bool, rowwise: bool = True,
               colwise: bool = True) -> NVFP4Tensor:
    import oracle
    q = NVFP4Tensor(M, N, swizzled=swizzled, row_scaled=row_scaled)
    if rowwise:
        q.data_row = torch.from_numpy(d["row_data"])
        rs = oracle.swizzle(d["row_scale"]) if swizzled else d["row_scale"].reshape(-1)
        q.scale_row = torch.from_numpy(np.ascontiguousarray(rs))
        q.amax_row = torch.from_numpy(d["amax_row"].copy())
    if colwise and not row_scaled:
        q.data_col = torch.from_numpy(d["col_data"])
        cs = oracle.swizzle(d["col_scale"]) if swizzled else d["col_scale"].reshape(-1)
        q.scale_col = torch.from_numpy(np.ascontiguousarray(cs))
        q.amax_col = torch.from_numpy(d["amax_col"].copy())
    return q


class OracleBackend:
    def local_amax(self, x, mode, sign_mask):
        import oracle
        xb = _bits(x)
        a = oracle.amax(xb)
        return torch.tensor([a, oracle.rht_amax(xb, sign_mask) if mode == "rht" else a], dtype=torch.float32)

    def cast(self, x, mode, amax, rowwise, colwise, swizzled, sign_mask, rbits=None):
        import oracle
        d = oracle.quantize(mode, _bits(x), rowwise, colwise, sign_mask=sign_mask,
                            amax=(float(amax[0]), float(amax[1])),
                            rbits=None if rbits is None else rbits.contiguous().numpy())
        return _to_tensor(d, x.shape[0], x.shape[1], swizzled, False, rowwise, colwise)

    def quantize_rows(self, x, swizzled):
        import oracle
        d = oracle.quantize("row_scaled", _bits(x), True, False)
        return _to_tensor(d, x.shape[0], x.shape[1], swizzled, True, True, False)


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CASES = [("1d", False), ("1d", True), ("2d", True), ("rht", False), ("row_scaled", True), ("row_scaled", False)]
SR_CASES = [("1d", True), ("2d", False)]


def _make_input(mode: str, M: int, N: int) -> torch.Tensor:
    if mode == "rht":
        return inputs.outliers(M, N, seed=61, frac=0.01, value=50.0)
    if mode == "row_scaled":
        return inputs.row_mix(M, N, seed=62, frac=0.05)
    return inputs.randn(M, N, seed=63)


def _rank_main(rank, world, port, outdir, scenario):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    results = {}
    try:
        if scenario == "parity":
            M, N = 384, 256
            for mode, swz in CASES:
                x = _make_input(mode, M, N)
                a, b = slab_bounds(M, world, rank, slab_alignment(mode, mode != "row_scaled", swz))
                q = quantize_slab(x[a:b].contiguous(), mode, colwise=mode != "row_scaled", swizzled=swz,
                                  sign_mask=inputs.sign_mask_from_seed(3), backend=OracleBackend())
                results[(mode, swz)] = {k: (None if getattr(q, k) is None else getattr(q, k).numpy())
                                        for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col",
                                                  "amax_col")} | {"M": q.M}
            rb = inputs.random_bytes(M, N, seed=64)
            for mode, swz in SR_CASES:
                x = _make_input(mode, M, N)
                a, b = slab_bounds(M, world, rank, slab_alignment(mode, True, swz))
                q = quantize_slab(x[a:b].contiguous(), mode, swizzled=swz, backend=OracleBackend(),
                                  rbits_local=rb[a:b].contiguous())
                results[("sr", mode, swz)] = {k: getattr(q, k).numpy() for k in
                                              ("data_row", "scale_row", "amax_row", "data_col", "scale_col",
                                               "amax_col")} | {"M": q.M}
        elif scenario == "bad_slab":
            x = inputs.randn(64, 64, seed=5)
            part = x[:40] if rank == 1 else x[:32]  # rank 1: 40 rows, not a multiple of 16
            try:
                quantize_slab(part.contiguous(), "1d", backend=OracleBackend())
                results["raised"] = None
            except ShardError as e:
                results["raised"] = str(e)
        elif scenario == "rank_exits":
            if rank == 1:
                os._exit(0)  # leaves without joining the exchange
            try:
                quantize_slab(inputs.randn(32, 32, seed=6), "1d", backend=OracleBackend())
                results["raised"] = None
            except ShardError as e:
                results["raised"] = "ShardError: " + str(e)
            except Exception as e:  # the collective's own error (peer gone)
                results["raised"] = type(e).__name__
    finally:
        with open(os.path.join(outdir, f"rank{rank}.pkl"), "wb") as f:
            pickle.dump(results, f)
        if scenario != "rank_exits":
            dist.destroy_process_group()


def _spawn(scenario, tmp_path, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path), scenario)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        if p.is_alive():
            p.kill()
            p.join()
            pytest.fail(f"rank process of scenario {scenario} did not finish")
    out = []
    for r in range(world):
        path = os.path.join(str(tmp_path), f"rank{r}.pkl")
        out.append(pickle.load(open(path, "rb")) if os.path.exists(path) else None)
    return out


def test_gloo_two_ranks_match_one_call_on_the_whole_tensor(tmp_path, oracle_mod):
    parts = _spawn("parity", tmp_path)
    M, N = 384, 256
    for mode, swz in CASES:
        pieces = []
        for r in range(2):
            d = parts[r][(mode, swz)]
            q = NVFP4Tensor(d["M"], N, swizzled=swz, row_scaled=mode == "row_scaled")
            for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
                setattr(q, k, None if d[k] is None else torch.from_numpy(d[k]))
            pieces.append(q)
        whole = assemble(pieces)
        x = _make_input(mode, M, N)
        ref = OracleBackend()
        if mode == "row_scaled":
            exp = ref.quantize_rows(x, swz)
        else:
            a = ref.local_amax(x, mode, inputs.sign_mask_from_seed(3))
            exp = ref.cast(x, mode, a, True, True, swz, inputs.sign_mask_from_seed(3))
        for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
            e, g = getattr(exp, k), getattr(whole, k)
            assert (e is None) == (g is None), (mode, swz, k)
            if e is not None:
                np.testing.assert_array_equal(g.numpy(), e.numpy(), err_msg=f"{mode} swizzled={swz} {k}")


def test_gloo_two_ranks_stochastic_rounding_matches_one_call(tmp_path, oracle_mod):
    """Each rank rounds its slab with the matching rows of the random bytes:
    the assembled result is the whole tensor's stochastic rounding."""
    parts = _spawn("parity", tmp_path)
    M, N = 384, 256
    rb = inputs.random_bytes(M, N, seed=64)
    for mode, swz in SR_CASES:
        pieces = []
        for r in range(2):
            d = parts[r][("sr", mode, swz)]
            q = NVFP4Tensor(d["M"], N, swizzled=swz)
            for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
                setattr(q, k, torch.from_numpy(d[k]))
            pieces.append(q)
        whole = assemble(pieces)
        x = _make_input(mode, M, N)
        ref = OracleBackend()
        exp = ref.cast(x, mode, ref.local_amax(x, mode, 0), True, True, swz, 0, rbits=rb)
        for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
            np.testing.assert_array_equal(getattr(whole, k).numpy(), getattr(exp, k).numpy(),
                                          err_msg=f"sr {mode} swizzled={swz} {k}")
        assert not np.array_equal(exp.data_row.numpy(), ref.cast(x, mode, ref.local_amax(x, mode, 0), True, True,
                                                                  swz, 0).data_row.numpy())


def test_gloo_invalid_slab_raises_on_every_rank(tmp_path):
    res = _spawn("bad_slab", tmp_path)
    assert res[0]["raised"] == "another rank's slab failed"
    assert res[1]["raised"].startswith("this rank's slab failed")


def test_gloo_rank_that_exits_makes_the_survivor_fail_not_hang(tmp_path):
    res = _spawn("rank_exits", tmp_path)
    assert res[0] is not None and res[0]["raised"] is not None
    assert res[1] is None or res[1] == {}


# ---------------------------------------------------------------------------
# GPU: ranks as host threads over slabs on one GPU
# ---------------------------------------------------------------------------

class _HostMax:
    """MAX of the ranks' exchange vectors on the host (a barrier between
    threads; the GPU kernels never wait on one another)."""

    def __init__(self, world):
        self.world, self.vals, self.lock = world, [], threading.Lock()
        self.bar = threading.Barrier(world, timeout=60)

    def __call__(self, v):
        with self.lock:
            self.vals.append(v.cpu())
        self.bar.wait()
        m = torch.stack(self.vals).max(0).values
        self.bar.wait()
        return m.to(v.device)


@pytest.mark.gpu
@pytest.mark.parametrize("mode,swz", [("1d", True), ("2d", True), ("rht", False), ("1d", False), ("row_scaled", True)])
def test_gpu_thread_ranks_match_one_call(mode, swz):
    import nvfp4_block_scaled_amax_gb300 as nv
    M, N, world = 1024, 512, 3
    x = _make_input(mode, M, N).cuda()
    mask = inputs.sign_mask_from_seed(3)
    exch = _HostMax(world)
    parts, errs = [None] * world, []

    def run(r):
        try:
            a, b = slab_bounds(M, world, r, slab_alignment(mode, mode != "row_scaled", swz))
            parts[r] = quantize_slab(x[a:b].contiguous(), mode, colwise=mode != "row_scaled", swizzled=swz,
                                     sign_mask=mask, exchange=exch)
            torch.cuda.current_stream().synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    whole = assemble(parts)
    exp = nv.quantize(x, mode, colwise=mode != "row_scaled", swizzled=swz, sign_mask=mask)
    torch.cuda.synchronize()
    for k in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
        e, g = getattr(exp, k), getattr(whole, k)
        assert (e is None) == (g is None), k
        if e is not None:
            assert torch.equal(g, e), (mode, swz, k)
