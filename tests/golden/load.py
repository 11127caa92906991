"""Reader for the small text fixtures in this folder (``key value value ...`` lines)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    out = {}
    with open(os.path.join(HERE, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            nums = [float(x) for x in vals]
            out[key] = nums[0] if len(nums) == 1 else nums
    return out
