"""Host-side logic of bench.py without a GPU: the max-over-ranks reduction and
the whole-job aggregate across a world of two gloo ranks, the kernel-source
hash that invalidates stored ncu traffic, and the derived integer-pipe peak."""
import importlib.util
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    b = _bench()
    d = b.Dist(world)
    # rank r "ran" 100 * (r + 1) rows in 1.5 + r seconds
    t = d.max(1.5 + rank)
    rows = d.max(100.0 * (rank + 1))  # the largest share, to check the reduction
    d.barrier()
    d.close()
    q.put((rank, t, rows))


def test_two_rank_gloo_reduction_and_aggregate():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]  # every rank sees the slowest rank's time
    assert [g[2] for g in got] == [200.0, 200.0]
    b = _bench()
    assert b.aggregate([100.0, 200.0], [1.5, 2.5]) == pytest.approx(120.0)


def test_kernel_source_hash_tracks_sources(tmp_path, monkeypatch):
    b = _bench()
    h = b.kernel_source_hash()
    assert len(h) == 16 and h == b.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "p.md").write_text("kernel_source_hash: %s\ndram_bytes_per_launch: 1000\n"
                               "captured_rows: 10\n" % h)
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    # ROOT now points at a folder without the sources: the hash no longer matches
    with pytest.raises(OSError):
        b.kernel_source_hash()


def test_stored_traffic_is_scaled_and_nulled_on_source_change(tmp_path, monkeypatch):
    b = _bench()
    h = b.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "p.md").write_text("kernel_source_hash: %s\ndram_bytes_per_launch: 1000\n"
                               "captured_rows: 10\n" % h)
    (prof / "q.md").write_text("kernel_source_hash: 0000000000000000\n"
                               "dram_bytes_per_launch: 1000\ncaptured_rows: 10\n")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    monkeypatch.setattr(b, "kernel_source_hash", lambda: h)
    assert b.ncu_traffic("p.md", 30) == pytest.approx(3000.0)
    assert b.ncu_traffic("q.md", 30) is None
    assert b.ncu_traffic("missing.md", 30) is None


def test_recorded_block_count_is_scaled_and_nulled_on_source_change(tmp_path, monkeypatch):
    b = _bench()
    h = b.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "p.md").write_text("kernel_source_hash: %s\ndram_bytes_per_launch: 1000\n"
                               "philox_blocks_per_launch: 640\ncaptured_rows: 10\n"
                               "philox_count_rows: 5\n" % h)
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    monkeypatch.setattr(b, "kernel_source_hash", lambda: h)
    assert b.profile_figure("p.md", "philox_blocks_per_launch", 20) == pytest.approx(1280.0)
    assert b.profile_figure("p.md", "philox_blocks_per_launch", 20,
                            rows_key="philox_count_rows") == pytest.approx(2560.0)
    assert b.profile_figure("p.md", "not_recorded", 20) is None
    monkeypatch.setattr(b, "kernel_source_hash", lambda: "0" * 16)
    assert b.profile_figure("p.md", "philox_blocks_per_launch", 20) is None


def test_headline_config_is_shared_by_both_arms():
    b = _bench()
    import workloads as W

    batch = W.Batch("t", np.zeros((4, 8), np.uint16), W.BF16, np.ones(4, np.float32),
                    np.zeros(4, np.uint64), np.zeros(4, np.uint64))
    c = b.headline_config(batch, 2)
    assert set(c) == {"workload", "global_batch", "vocab"}
    assert c["global_batch"] == 8 and c["vocab"] == 8


def test_side_workload_needs_quick(monkeypatch):
    b = _bench()
    monkeypatch.setattr("sys.argv", ["bench.py", "--quick", "--workload", "sweep", "--batch", "8"])
    a = b.parse_args()
    assert (a.workload, a.batch, a.vocab, a.categorical) == ("sweep", 8, 151936, False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--workload", "hlg"])
    with pytest.raises(SystemExit):
        b.parse_args()  # a side case never replaces the headline line
    monkeypatch.setattr("sys.argv", ["bench.py", "--categorical"])
    with pytest.raises(SystemExit):
        b.parse_args()


def test_cpu_model_names_the_host():
    b = _bench()
    name = b.cpu_model()
    assert isinstance(name, str) and name


def test_kernel_source_hash_covers_the_headline_kernel_only(tmp_path, monkeypatch):
    import shutil

    b = _bench()
    csrc = os.path.join(ROOT, "token_sampling_logits_gb300", "csrc")
    copy = tmp_path / "token_sampling_logits_gb300" / "csrc"
    shutil.copytree(csrc, copy)
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    h = b.kernel_source_hash()
    with open(copy / "gsample_hlg.cu", "a") as f:
        f.write("\n// another kernel's change\n")
    assert b.kernel_source_hash() == h
    with open(copy / "gsample_sample.cu", "a") as f:
        f.write("\n// the headline kernel's change\n")
    assert b.kernel_source_hash() != h
