"""The bench's algorithmic byte count (the roofline's numerator) against an independent
count from the model's tensor list: every matrix streamed once per step, the embedding
rows a step reads, and the keys/values of each slot's window."""
import numpy as np

import bench
import synth


def _independent(s, lens):
    wb = 2 if s.weight_dtype == "bf16" else 4
    kvb = 2 if s.kv_dtype == "bf16" else 4
    streamed = 0
    for name, shape, init in synth.weight_specs(s):
        if init == "gain" or name.startswith(("emb.", "dep.emb.")):
            continue  # gains stay in L1/L2; embeddings are read one row per token
        streamed += int(np.prod(shape)) * wb
    rows = (1 + s.n_q) * s.d * wb + s.dep_steps * s.dep_d * wb  # 17 embedding rows + 16 depformer rows
    kv_pos = s.n_layers * 2 * s.d * kvb  # one position's key and value over all layers
    return streamed + sum(rows + ln * kv_pos + kv_pos for ln in lens)


def test_algorithmic_bytes_match_the_tensor_list():
    s = synth.FULL
    for lens in ([256], [3000] * 8, [0, 17, 2999]):
        assert bench.algorithmic_bytes(s, lens) == _independent(s, lens)
    # the full shape streams 16.08 GB of weights per step
    assert abs(bench.algorithmic_bytes(s, []) - 16_083_058_688) == 0
