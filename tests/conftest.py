import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    import torch

    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def switches():
    """Sets the library's test switches (kernel choice, compact Q tile) through
    pa_set_switch, and puts back the values they had when the test ends."""
    import paged_kv_attention_08_gb300 as pa

    names = {"kernel": pa.SWITCH_MULTI_KERNEL, "compact_q": pa.SWITCH_TILE_COMPACT_Q}
    kernels = {"auto": pa.KERNEL_AUTO, "mma": pa.KERNEL_MMA, "tile": pa.KERNEL_TILE}
    saved = {w: pa.get_switch(w) for w in names.values()}

    def set_(kernel=None, compact_q=None):
        if kernel is not None:
            pa.set_switch(names["kernel"], kernels[kernel])
        if compact_q is not None:
            pa.set_switch(names["compact_q"], int(compact_q))

    yield set_
    for w, v in saved.items():
        pa.set_switch(w, v)
