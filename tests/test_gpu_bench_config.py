"""Full-size parity in the launch configuration bench.py times: the layer-stack workload's
layers at T=4096 and batch-1 decode, replayed from CUDA graphs, checked against the oracle on
sampled tokens (each token's output depends only on that token, so the oracle computes the
sampled rows alone)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
import oracle as O  # noqa: E402
from synthetic import FULL, make_layer, make_tokens  # noqa: E402
from tests import moe_check as C  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bench_launch_configuration_sampled():
    args = bench.parse_args(["--layers", "2", "--prefill-tokens", "4096", "--decode-steps", "3"])
    from quantized_grouped_gemm_router_gb300 import build as B
    B.build()
    W = bench.Workload(args, torch.device("cuda", 0))
    run_pre, run_dec = bench.capture(W, graphs=True)
    for _ in range(2):   # replay twice: counters and accumulators must be reset by each call
        run_pre()
        run_dec()
    torch.cuda.synchronize()
    assert W.m.read_device_status(W.ws_p) == 0 and W.m.read_device_status(W.ws_d) == 0
    rng = np.random.default_rng(0)
    for l in range(args.layers):
        npl = make_layer(FULL, seed=l)
        xp = make_tokens(4096, FULL.d, seed=l, stream=1)
        rows = np.sort(rng.choice(4096, size=24, replace=False))
        rows[0], rows[-1] = 0, 4095
        ref = O.moe_forward(xp[rows], npl, tile_rows=256)["y"]
        got = C.bf16_bits_f64(W.yp[l][torch.as_tensor(rows, device="cuda")])
        C.check_y(got, ref, f"prefill layer {l}")
        xd = make_tokens(args.decode_steps * args.layers, FULL.d, seed=0, stream=2).reshape(
            args.decode_steps, args.layers, FULL.d)
        for s in range(args.decode_steps):
            ref = O.moe_forward(xd[s, l][None], npl, tile_rows=256)["y"]
            C.check_y(C.bf16_bits_f64(W.yd[s, l][None]), ref, f"decode step {s} layer {l}")
