"""The gather's source check accepts device memory however torch allocated it.

kvsel_compact refuses a source that the device cannot read (cudaPointerGetAttributes decides).
Memory from torch's expandable segments (virtual-memory mappings) and from the stream-ordered
allocator (cudaMallocAsync pools) is device memory too: a step run with either allocator must
gather exactly the rows torch's own indexing gathers.  Each allocator is chosen at start-up, so
each case runs in a child process.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
from attention_kv_cache_gb300 import kvsel as K
from attention_kv_cache_gb300 import synth as S
from attention_kv_cache_gb300.pipeline import Pipeline, pack

dev = torch.device("cuda:0")
w = S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[3000])
inp = S.make_inputs(w, "cpu")
q, k, v = pack(inp, dev)
pipe = Pipeline(w, dev)
pipe.run(q, k, v)
torch.cuda.synchronize()
assert K.kvsel_read_device_error(pipe.ws) == K.OK
n = w.prefix_lens[0] + w.window
kk = k.view(w.n_layers, w.h_kv, n, w.head_dim)
vv = v.view(w.n_layers, w.h_kv, n, w.head_dim)
idx = pipe.idx[0].long()
for l in range(w.n_layers):
    for g in range(w.h_kv):
        assert torch.equal(pipe.k_out[0, l, g], kk[l, g, idx[l, g]])
        assert torch.equal(pipe.v_out[0, l, g], vv[l, g, idx[l, g]])
print("gathered rows equal")
"""


@pytest.mark.parametrize("conf", ["expandable_segments:True", "backend:cudaMallocAsync"])
def test_gather_from_each_allocator(conf, cuda):
    env = dict(os.environ, PYTORCH_CUDA_ALLOC_CONF=conf)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "gathered rows equal" in r.stdout
