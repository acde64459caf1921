"""Host-side pieces of the bench on CPU: the clock sampler's reading of
nvidia-smi lines (only samples taken under load count, throttle reasons are
collected) and the rule that an ncu traffic figure is reported only while the
kernel's sources match the capture."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, mx=2070, power=900.0, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {mx}, {power}, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}"


def _sampler(lines, first):
    s = bench.ClockSampler(0)
    s.lines = list(lines)
    s.first = first
    return s


def _stats(s):
    # stop() without a process: the parsing part only
    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    class _T:
        def join(self, timeout=None):
            pass

    s.proc, s.thread = _P(), _T()
    return s.stop()


def test_idle_samples_before_the_load_are_dropped():
    got = _stats(_sampler([_line(345), _line(2070), _line(2055), _line(2070)], first=1))
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070
    assert got["sm_max_mhz"] == 2070
    assert got["reasons"] == []


def test_all_samples_used_when_none_landed_under_load():
    got = _stats(_sampler([_line(1980)], first=1))
    assert got["samples"] == 1 and got["sm_mhz"] == 1980


def test_throttle_reasons_are_collected():
    got = _stats(_sampler([_line(2070, cap="Active"), _line(1800, hwt="Active")], first=0))
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_malformed_lines_are_skipped():
    got = _stats(_sampler(["garbage", _line(2070), "0, [N/A], 2070, 1, 0, a, b, c, d"], first=0))
    assert got["samples"] == 1


def test_traffic_reported_only_for_matching_sources(tmp_path, monkeypatch):
    from normalization_layernorm_rmsnorm_gb300.build import source_digest
    files = ["common.cuh", "libnorm.h"]
    prof = tmp_path / "profiles"
    prof.mkdir()
    data = {
        "k_ok": {"dram_bytes_per_launch": 123, "sources": files, "source_digest": source_digest(files)},
        "k_stale": {"dram_bytes_per_launch": 456, "sources": files, "source_digest": "0" * 16},
        "k_nodigest": {"dram_bytes_per_launch": 789, "sources": files},
    }
    (prof / "ncu_traffic.json").write_text(json.dumps(data))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k_ok") == 123
    assert bench.ncu_traffic("k_stale") is None
    assert bench.ncu_traffic("k_nodigest") is None
    assert bench.ncu_traffic("missing") is None


def test_e2e_plan_uploads_first_reads_and_downloads_last_writes():
    # a forward writing y and the saved mean, then a backward reading them with
    # dy: x, w and dy come from the host before the call that first reads them,
    # the saved mean (written by the forward) is not uploaded again; y and mean
    # are downloaded after the forward, dx and dw after the backward
    import types
    x, w, y, mean, dy, dx, dw = (object() for _ in range(7))
    fwd = types.SimpleNamespace(inputs=[x, w], outputs=[y, mean])
    bwd = types.SimpleNamespace(inputs=[dy, x, w, mean], outputs=[dx, dw])
    up, down = bench.e2e_plan([fwd, bwd])
    assert up[0] == [x, w] and up[1] == [dy]
    assert down[0] == [y, mean] and down[1] == [dx, dw]


def test_e2e_plan_rewritten_tensor_moves_once_each_way():
    # running statistics read and updated by two calls: uploaded before the
    # first, downloaded after the last
    import types
    rm = object()
    a = types.SimpleNamespace(inputs=[rm], outputs=[rm])
    b = types.SimpleNamespace(inputs=[rm], outputs=[rm])
    up, down = bench.e2e_plan([a, b])
    assert up[0] == [rm] and 1 not in up
    assert down[1] == [rm] and 0 not in down
