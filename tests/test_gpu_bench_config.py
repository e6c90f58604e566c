"""Full-size parity in the launch configuration bench.py times: the whole layer-stack workload
(40 layers at T=4096, 256 batch-1 decode steps through the 40 layers), replayed from CUDA graphs,
checked against the oracle on layers 0, 19 and 39 (sampled prefill tokens; decode steps 0, 127
and 255). Each token's output depends only on that token, so the oracle computes the sampled
rows alone."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
import oracle as O  # noqa: E402
from synthetic import FULL, make_layer, make_tokens  # noqa: E402
from tests import moe_check as C  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bench_launch_configuration_sampled():
    args = bench.parse_args(["--layers", "40", "--prefill-tokens", "4096", "--decode-steps", "256"])
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
    xd = make_tokens(args.decode_steps * args.layers, FULL.d, seed=0, stream=2).reshape(
        args.decode_steps, args.layers, FULL.d)
    for l in (0, 19, 39):
        npl = make_layer(FULL, seed=l)
        xp = make_tokens(4096, FULL.d, seed=l, stream=1)
        rows = np.sort(rng.choice(4096, size=24, replace=False))
        rows[0], rows[-1] = 0, 4095
        ref = O.moe_forward(xp[rows], npl, tile_rows=256)["y"]
        got = C.bf16_bits_f64(W.yp[l][torch.as_tensor(rows, device="cuda")])
        C.check_y(got, ref, f"prefill layer {l}")
        for s in (0, 127, 255):
            ref = O.moe_forward(xd[s, l][None], npl, tile_rows=256)["y"]
            C.check_y(C.bf16_bits_f64(W.yd[s, l][None]), ref, f"decode step {s} layer {l}")
