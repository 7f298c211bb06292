"""bench.py's oracle arm (--impl reference) runs on the host alone: it must
print its JSON line without ever loading the CUDA library, so that its timing
is independent of the product path.  The one-core child used for the
single-core oracle figure runs the same host cycle."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import runpy, sys
sys.argv = ['bench.py'] + sys.argv[1:]
runpy.run_path('bench.py', run_name='__main__')
maps = open('/proc/self/maps').read()
print('LIBDFLASH_LOADED=%d' % ('libdflash' in maps))
"""


def test_reference_arm_never_loads_the_library():
    r = subprocess.run([sys.executable, "-c", PROBE, "--impl", "reference", "--workload", "0",
                        "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    line = json.loads(lines[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert "LIBDFLASH_LOADED=0" in r.stdout


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "0",
                        "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_one_core_oracle_child():
    sys.path.insert(0, ROOT)
    import bench
    out = bench.one_core_oracle(0, timeout_s=300)
    assert "seconds" in out, out
    assert out["cores"] == 1 and out["seconds"] > 0
