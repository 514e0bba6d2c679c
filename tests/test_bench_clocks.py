"""The benchmark's clock sampler against a stand-in nvidia-smi (a shell script
on PATH), so that its parsing runs without a GPU: samples inside the timed
region, throttle reasons, and the instantaneous power reading when the tool
knows that field (and the averaged one when it does not)."""

import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FAKE = r"""#!/bin/bash
# Stand-in for nvidia-smi: a single query of power.draw.instant prints one
# number (or fails when KNOW_INSTANT=0); a looping query prints rows.
args="$*"
if [[ "$args" != *"-lms"* ]]; then
  if [[ "$KNOW_INSTANT" == "1" ]]; then echo "1234.50"; exit 0; fi
  echo 'Field "power.draw.instant" is not a valid field to query.' >&2; exit 2
fi
for i in 0 1 2 3 4 5; do
  ts=$(date +"%Y/%m/%d %H:%M:%S.%3N")
  reason="Not Active"; if [[ $i == 3 ]]; then reason="Active"; fi
  row="$ts, 0, $((1900 + i)), 2070, 600.00, 0x0000000000000000, Not Active, Not Active, Not Active, $reason"
  if [[ "$args" == *"power.draw.instant"* ]]; then row="$row, $((1000 + 50 * i)).25"; fi
  echo "$row"
  sleep 0.05
done
exec sleep 30
"""


def make_fake(tmp_path):
    p = tmp_path / "nvidia-smi"
    p.write_text(FAKE)
    p.chmod(p.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def sample(monkeypatch, tmp_path, know_instant):
    import bench

    monkeypatch.setenv("PATH", make_fake(tmp_path) + os.pathsep + os.environ["PATH"])
    monkeypatch.setenv("KNOW_INSTANT", "1" if know_instant else "0")
    s = bench.ClockSampler(0)
    s.mark("t0")
    s.start()
    time.sleep(0.3)
    s.mark("t1")
    return s.stop()


def test_sampler_reads_instant_power(monkeypatch, tmp_path):
    c = sample(monkeypatch, tmp_path, True)
    assert c["power_field"] == "power.draw.instant"
    assert c["samples"] == 6 and c["samples_in_timed_region"] == 6
    assert c["sm_max_mhz"] == 2070.0 and c["sm_mhz"] == 1902.5
    assert c["reasons"] == ["sw_power_cap"]
    assert c["power_w_max"] == 1250.25


def test_sampler_falls_back_to_averaged_power(monkeypatch, tmp_path):
    c = sample(monkeypatch, tmp_path, False)
    assert c["power_field"] == "power.draw"
    assert c["samples"] == 6
    assert c["power_w_max"] == 600.0
