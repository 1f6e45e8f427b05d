"""Host-side logic of bench.py and of the byte accounting, on the CPU:
the page-printed expert sizes, clock parsing, the max-over-ranks reduction
across two gloo ranks, and the reference (oracle) arm's JSON line."""
import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "page_numbers.json")


def test_accounting_matches_page_numbers():
    from mixture_experts_routed_softmax_gb300 import accounting as acc
    g = json.load(open(GOLDEN))
    eb = g["expert_bytes_bf16"]
    assert acc.expert_bytes(eb["d"], eb["f"]) == eb["value_mib"] * 2 ** 20
    rs = g["routed_expert_set"]
    total = acc.expert_bytes(eb["d"], eb["f"]) * rs["experts"] * rs["layers"] / 2 ** 30
    assert abs(total - rs["value_gib"]) <= rs["tolerance_gib"]
    dc = g["decode_copies"]
    assert acc.expert_bytes(eb["d"], eb["f"]) * dc["copies"] == dc["value_mib"] * 2 ** 20
    de = g["distinct_experts"]
    assert abs(acc.expected_active_experts(de["E"], de["k"], de["T"]) - de["value"]) <= de["tolerance"]


def test_kernel_costs_add_up_to_the_layer_formula():
    from mixture_experts_routed_softmax_gb300 import accounting as acc
    s = acc.Shape(T=16384, d=2880, f=2880, E=32, k=4, E_active=32)
    F, B = acc.totals(s)
    P = s.T * s.k
    fwd_expert = 6 * P * s.d * s.f
    assert F >= 3 * fwd_expert and F <= 3 * fwd_expert + 10 * s.T * s.d * s.E
    fw_f, _ = acc.totals(s, backward=False)
    assert fw_f == fwd_expert + 2 * s.T * s.d * s.E
    assert B > 3 * acc.expert_bytes(s.d, s.f) * s.E


def test_clock_rows_parse():
    import bench
    rows = [["0", "1900 MHz", "2070 MHz", "900 W", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "1940 MHz", "2070 MHz", "950 W", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "1960 MHz", "2070 MHz", "960 W", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    c = bench.parse_clock_rows(rows)
    # under load = power in the upper half of the range seen (950 W and 960 W here)
    assert c["sm_mhz"] == 1950.0 and c["samples_under_load"] == 2
    assert c["sm_mhz_all_samples"] == 1940.0 and c["samples"] == 3
    assert c["sm_max_mhz"] == 2070.0 and c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_rows([]) is None


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    out[rank] = bench.max_over_ranks(10.0 + rank)
    bench.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == 11.0 and out[1] == 11.0


def test_reference_arm_prints_one_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1", "--ref-tokens", "8"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_decode_costs_match_the_forward_arithmetic():
    from mixture_experts_routed_softmax_gb300 import accounting as acc
    s = acc.Shape(T=8, d=2048, f=768, E=128, k=8, E_active=52)
    fl, by = acc.decode_costs(s)
    assert fl == acc.totals(s, backward=False)[0]       # the same products, one launch
    w = 3 * 52 * 2048 * 768 * 2
    assert w < by < w + 2 * 2**20                       # weights dominate; the rest is small


def test_fused_forward_costs_drop_only_the_kept_activations():
    """The fused inference forward moves the five-call forward's bytes less
    the G and U rows it keeps in tensor memory (2 P f in the bf16 layout),
    with the same FLOPs: 6 P d f for the experts plus the router's."""
    from mixture_experts_routed_softmax_gb300 import accounting as acc
    s = acc.Shape(T=8192, d=2048, f=768, E=128, k=8, E_active=128)
    five = acc.kernel_costs(s, backward=False)
    fused = acc.fused_forward_costs(s)
    f5 = sum(c[0] for c in five.values())
    ff = sum(c[0] for c in fused.values())
    b5 = sum(c[1] for c in five.values())
    bf = sum(c[1] for c in fused.values())
    assert ff == f5 == 6 * s.P * s.d * s.f + 2 * s.T * s.d * s.E
    assert b5 - bf == 2 * s.P * s.f * 2
    assert set(fused) == {"router_logits", "topk", "permute", "fused_fwd", "combine"}
